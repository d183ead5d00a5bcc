"""Pins of the fp64 oracle to things other than itself (CPU only).

Each check is chosen so that a plausible mistake in the oracle -- a dropped
term, a wrong sign, a wrong mask index, a transposed operand, natural vs base-2
log -- fails at least one of them:

* hand-derived closed forms (tests/golden/closed_form_cases.json);
* torch's own float64 SDPA and autograd on the CPU (library special case;
  torch's ``is_causal`` is the top-left mask the pages ask for);
* an independent full-matrix numpy softmax for tiny problems;
* central finite differences of L = sum(O * dO) for the backward;
* invariants: rows of P sum to 1, causal row 0, Q = 0 prefix mean, the
  gradient identities, and layout equivalences between dense and THD.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import sdpa_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_form_cases.json")


def _rel(a, b):
    """max|a-b| over max(max|b|, 1): relative for O(1) tensors, absolute near 0."""
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1.0))


# ---------------------------------------------------------------- closed forms
@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_closed_form_cases(case):
    q, k, v, do = (np.array(case[x], np.float64)[None, None] for x in ("q", "k", "v", "dout"))
    o, lse = oracle.sdpa_fwd(q, k, v, case["scale"], case["causal"])
    np.testing.assert_allclose(o[0, 0], case["o"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse[0, 0], case["lse"], rtol=0, atol=1e-14)
    dq, dk, dv = oracle.sdpa_bwd(q, k, v, do, case["scale"], case["causal"])
    np.testing.assert_allclose(dq[0, 0], case["dq"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(dk[0, 0], case["dk"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(dv[0, 0], case["dv"], rtol=0, atol=1e-14)


# ---------------------------------------------------- torch float64 reference
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("s_q,s_kv", [(37, 37), (20, 45), (45, 20), (1, 9)])
def test_against_torch_float64(causal, s_q, s_kv):
    g = torch.Generator().manual_seed(7 + s_q * 3 + s_kv)
    b, h, d = 2, 3, 16
    q = torch.randn(b, h, s_q, d, generator=g, dtype=torch.float64, requires_grad=True)
    k = torch.randn(b, h, s_kv, d, generator=g, dtype=torch.float64, requires_grad=True)
    v = torch.randn(b, h, s_kv, d, generator=g, dtype=torch.float64, requires_grad=True)
    do = torch.randn(b, h, s_q, d, generator=g, dtype=torch.float64)
    scale = 0.37
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=scale)
    ref.backward(do)
    scores = scale * q.detach() @ k.detach().transpose(-1, -2)
    if causal:
        allowed = torch.ones(s_q, s_kv, dtype=torch.bool).tril()
        scores = scores.masked_fill(~allowed, float("-inf"))
    lse_ref = torch.logsumexp(scores, dim=-1)

    o, lse = oracle.sdpa_fwd(q.detach(), k.detach(), v.detach(), scale, causal)
    dq, dk, dv = oracle.sdpa_bwd(q.detach(), k.detach(), v.detach(), do, scale, causal)
    assert _rel(o, ref.detach().numpy()) < 1e-13
    np.testing.assert_allclose(lse, lse_ref.numpy(), rtol=0, atol=1e-12)
    assert _rel(dq, q.grad.numpy()) < 1e-12
    assert _rel(dk, k.grad.numpy()) < 1e-12
    assert _rel(dv, v.grad.numpy()) < 1e-12


# --------------------------------------------- independent numpy brute force
def _brute(q, k, v, do, scale, causal):
    """Full-matrix softmax attention written out in numpy (independent code)."""
    s = scale * np.einsum("id,jd->ij", q, k)
    n_q, n_kv = s.shape
    mask = np.ones_like(s, dtype=bool)
    if causal:
        mask = np.arange(n_kv)[None, :] <= np.arange(n_q)[:, None]
    s = np.where(mask, s, -np.inf)
    mx = s.max(axis=1, keepdims=True)
    e = np.where(mask, np.exp(s - mx), 0.0)
    p = e / e.sum(axis=1, keepdims=True)
    o = p @ v
    lse = (mx[:, 0] + np.log(e.sum(axis=1)))
    dp = do @ v.T
    dsum = (do * o).sum(axis=1, keepdims=True)
    ds = p * (dp - dsum)
    return o, lse, scale * ds @ k, scale * ds.T @ q, p.T @ do


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n_q,n_kv,d", [(1, 1, 1), (5, 5, 3), (16, 16, 8), (7, 13, 4), (13, 7, 5)])
def test_against_brute_force(causal, n_q, n_kv, d):
    rng = np.random.default_rng(n_q * 100 + n_kv * 10 + d)
    q, k, v = rng.normal(size=(n_q, d)), rng.normal(size=(n_kv, d)), rng.normal(size=(n_kv, d))
    do = rng.normal(size=(n_q, d))
    scale = 1.0 / math.sqrt(d)
    o_b, lse_b, dq_b, dk_b, dv_b = _brute(q, k, v, do, scale, causal)
    o, lse = oracle.sdpa_fwd(q[None, None], k[None, None], v[None, None], scale, causal)
    dq, dk, dv = oracle.sdpa_bwd(q[None, None], k[None, None], v[None, None], do[None, None],
                                 scale, causal)
    np.testing.assert_allclose(o[0, 0], o_b, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse[0, 0], lse_b, rtol=0, atol=1e-13)
    np.testing.assert_allclose(dq[0, 0], dq_b, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk[0, 0], dk_b, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv[0, 0], dv_b, rtol=0, atol=1e-12)


# ------------------------------------------------------- finite differences
@pytest.mark.parametrize("causal", [False, True])
def test_backward_finite_differences(causal):
    rng = np.random.default_rng(11)
    n, d = 8, 4
    q, k, v, do = (rng.normal(size=(1, 1, n, d)) for _ in range(4))
    scale = 0.6
    dq, dk, dv = oracle.sdpa_bwd(q, k, v, do, scale, causal)

    def loss(qq, kk, vv):
        return float((oracle.sdpa_fwd(qq, kk, vv, scale, causal)[0] * do).sum())

    eps = 1e-6
    for which, grad in ((0, dq), (1, dk), (2, dv)):
        num = np.zeros_like(grad)
        for idx in np.ndindex(*grad.shape):
            args = [q.copy(), k.copy(), v.copy()]
            args[which][idx] += eps
            lp = loss(*args)
            args[which][idx] -= 2 * eps
            lm = loss(*args)
            num[idx] = (lp - lm) / (2 * eps)
        assert _rel(grad, num) < 1e-6, which


# ----------------------------------------------------------------- invariants
def test_rows_sum_to_one():
    rng = np.random.default_rng(3)
    b, h, s, d = 1, 2, 33, 8
    q, k = rng.normal(size=(b, h, s, d)), rng.normal(size=(b, h, s, d))
    ones = np.ones((b, h, s, d))
    for causal in (False, True):
        o, _ = oracle.sdpa_fwd(q, k, ones, 0.5, causal)
        np.testing.assert_allclose(o, 1.0, rtol=0, atol=1e-14)


def test_causal_row0_and_lse():
    rng = np.random.default_rng(4)
    b, h, s, d = 2, 2, 17, 8
    q, k, v = (rng.normal(size=(b, h, s, d)) for _ in range(3))
    scale = 0.3
    o, lse = oracle.sdpa_fwd(q, k, v, scale, True)
    np.testing.assert_allclose(o[:, :, 0], v[:, :, 0], rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse[:, :, 0], scale * (q[:, :, 0] * k[:, :, 0]).sum(-1),
                               rtol=0, atol=1e-14)
    # LSE is the natural-log log-sum-exp of the scaled scores
    s_full = scale * np.einsum("bhid,bhjd->bhij", q, k)
    lse_direct = np.array([[[np.log(np.exp(s_full[bb, hh, i, :i + 1]).sum()) for i in range(s)]
                            for hh in range(h)] for bb in range(b)])
    np.testing.assert_allclose(lse, lse_direct, rtol=0, atol=1e-12)


def test_zero_query_gives_prefix_mean():
    rng = np.random.default_rng(5)
    b, h, s, d = 1, 3, 21, 6
    q = np.zeros((b, h, s, d))
    k, v = rng.normal(size=(b, h, s, d)), rng.normal(size=(b, h, s, d))
    o, lse = oracle.sdpa_fwd(q, k, v, 0.25, True)
    prefix_mean = np.cumsum(v, axis=2) / np.arange(1, s + 1)[None, None, :, None]
    np.testing.assert_allclose(o, prefix_mean, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, np.log(np.arange(1, s + 1))[None, None].repeat(h, 1),
                               rtol=0, atol=1e-13)
    o, lse = oracle.sdpa_fwd(q, k, v, 0.25, False)
    np.testing.assert_allclose(o, v.mean(axis=2, keepdims=True).repeat(s, 2), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, math.log(s), rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_gradient_identities(causal):
    rng = np.random.default_rng(6)
    b, h, s, d = 1, 2, 24, 8
    q, k, v, do = (rng.normal(size=(b, h, s, d)) for _ in range(4))
    scale = 0.35
    dq, dk, dv = oracle.sdpa_bwd(q, k, v, do, scale, causal)
    # rows of P sum to one  =>  sum_j dV_j = sum_i dO_i
    np.testing.assert_allclose(dv.sum(axis=2), do.sum(axis=2), rtol=0, atol=1e-12)
    # sum_i dQ_i.Q_i = sum_j dK_j.K_j = scale * sum_ij dS_ij Q_i.K_j
    np.testing.assert_allclose((dq * q).sum(axis=(2, 3)), (dk * k).sum(axis=(2, 3)),
                               rtol=0, atol=1e-11)
    # constant V => O = c and dS vanishes, so dQ = dK = 0
    c = np.broadcast_to(rng.normal(size=(1, 1, 1, d)), (b, h, s, d)).copy()
    o, _ = oracle.sdpa_fwd(q, k, c, scale, causal)
    np.testing.assert_allclose(o, c, rtol=0, atol=1e-13)
    dq, dk, dv = oracle.sdpa_bwd(q, k, c, do, scale, causal)
    assert np.abs(dq).max() < 1e-12 and np.abs(dk).max() < 1e-12


def test_dead_rows():
    """s_kv = 0: every row is dead -> O = 0, LSE = -inf, zero gradients."""
    q = np.ones((1, 1, 4, 8))
    k = np.zeros((1, 1, 0, 8))
    o, lse = oracle.sdpa_fwd(q, k, k, 0.5, True)
    assert np.all(o == 0) and np.all(np.isneginf(lse))
    dq, _, _ = oracle.sdpa_bwd(q, k, k, q, 0.5, True)
    assert np.all(dq == 0)


# ------------------------------------------------------- layout equivalences
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_equals_dense(causal):
    h, d, L, n = 3, 8, 19, 4
    q, k, v, do = sdpa_inputs.dense(n, h, L, L, d, seed=9, dtype=torch.float64)
    o_d, lse_d = oracle.sdpa_fwd(q, k, v, 0.3, causal)
    dq_d, dk_d, dv_d = oracle.sdpa_bwd(q, k, v, do, 0.3, causal)

    def pack(x):  # [n,h,L,d] -> [n*L,h,d]
        return x.permute(0, 2, 1, 3).reshape(n * L, h, d)

    cu = sdpa_inputs.cu_seqlens([L] * n)
    o_v, lse_v = oracle.sdpa_varlen_fwd(pack(q), pack(k), pack(v), cu, cu, 0.3, causal)
    dq_v, dk_v, dv_v = oracle.sdpa_varlen_bwd(pack(q), pack(k), pack(v), pack(do), cu, cu, 0.3,
                                              causal)
    unpack = lambda a: a.reshape(n, L, h, -1).transpose(0, 2, 1, 3)  # noqa: E731
    np.testing.assert_array_equal(unpack(o_v), o_d)
    np.testing.assert_array_equal(lse_v.reshape(n, L, h).transpose(0, 2, 1), lse_d)
    np.testing.assert_array_equal(unpack(dq_v), dq_d)
    np.testing.assert_array_equal(unpack(dk_v), dk_d)
    np.testing.assert_array_equal(unpack(dv_v), dv_d)


def test_varlen_mixed_lengths_per_sequence():
    """Each THD sequence equals its own dense problem (per-sequence reference)."""
    lens = [5, 0, 17, 1, 9]
    h, d = 2, 4
    q, k, v, do, cu, _ = sdpa_inputs.packed(lens, lens, h, d, seed=10, dtype=torch.float64)
    o, lse = oracle.sdpa_varlen_fwd(q, k, v, cu, cu, 0.5, True)
    dq, dk, dv = oracle.sdpa_varlen_bwd(q, k, v, do, cu, cu, 0.5, True)
    for n, L in enumerate(lens):
        a, e = int(cu[n]), int(cu[n + 1])
        sl = lambda x: x[a:e].permute(1, 0, 2)[None]  # noqa: E731
        o_r, lse_r = oracle.sdpa_fwd(sl(q), sl(k), sl(v), 0.5, True)
        g = oracle.sdpa_bwd(sl(q), sl(k), sl(v), sl(do), 0.5, True)
        np.testing.assert_array_equal(o[a:e], o_r[0].transpose(1, 0, 2))
        np.testing.assert_array_equal(lse[a:e], lse_r[0].T)
        for got, ref in zip((dq, dk, dv), g):
            np.testing.assert_array_equal(got[a:e], ref[0].transpose(1, 0, 2))


def test_row_sampled_entry_points_match_full():
    rng = np.random.default_rng(12)
    n, d = 40, 8
    q, k, v, do = (rng.normal(size=(n, d)) for _ in range(4))
    rows = np.array([0, 3, 39, 17], np.int32)
    o, lse = oracle.sdpa_fwd(q[None, None], k[None, None], v[None, None], 0.4, True)
    o_r, lse_r = oracle.attn_fwd_rows(q, k, v, rows, 0.4, True)
    np.testing.assert_array_equal(o_r, o[0, 0][rows])
    np.testing.assert_array_equal(lse_r, lse[0, 0][rows])
    dq, dk, dv = oracle.sdpa_bwd(q[None, None], k[None, None], v[None, None], do[None, None],
                                 0.4, True)
    kv_rows = np.array([1, 38, 20], np.int32)
    dq_r, dk_r, dv_r = oracle.attn_bwd_rows(q, k, v, do, rows, kv_rows, 0.4, True)
    np.testing.assert_array_equal(dq_r, dq[0, 0][rows])
    np.testing.assert_array_equal(dk_r, dk[0, 0][kv_rows])
    np.testing.assert_array_equal(dv_r, dv[0, 0][kv_rows])


# -------------------------------------------------------------- input recipe
def test_inputs_are_seeded_and_exact():
    a = sdpa_inputs.dense(1, 2, 8, 8, 4, seed=1)
    b = sdpa_inputs.dense(1, 2, 8, 8, 4, seed=1)
    for x, y in zip(a, b):
        assert torch.equal(x, y) and x.dtype == torch.bfloat16
    q1, k1, _, _ = sdpa_inputs.dense(1, 1, 8, 8, 4, seed=3)
    q2, k2, _, _ = sdpa_inputs.dense(1, 1, 8, 8, 4, seed=3, qk_mult=2.0)
    assert torch.equal(q2.float(), 2 * q1.float()) and torch.equal(k2.float(), 2 * k1.float())
    lens = sdpa_inputs.varlen_lengths(16, 2004)
    assert len(lens) == 16 and all(64 <= L <= 4096 for L in lens)
    cu = sdpa_inputs.cu_seqlens(lens)
    assert cu.dtype == torch.int32 and int(cu[-1]) == sum(lens) and int(cu[0]) == 0
