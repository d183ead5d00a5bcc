"""Pins for the oracle's extended masks (bottom-right causal, left window) and
grouped key/value heads, against references that are not the oracle:

- torch's float64 scaled_dot_product_attention with an explicit boolean mask
  and repeated K/V heads, plus autograd for the gradients (library case);
- an independent numpy full-matrix softmax (brute force, tiny sizes);
- central finite differences of sum(O * dO);
- closed forms: a window of 0 keys under a causal mask leaves one key per row,
  so O_i = V_{i+delta} and LSE_i = scale * Q_i . K_{i+delta}; rows that see no
  key (bottom-right with s_q > s_kv) give O = 0 and LSE = -inf.

Mask semantics (cudnn-frontend PR #554 `sdpa` op, `causal_bottom_right` and
`window_left`): delta = s_kv - s_q for bottom-right, else 0; a causal mask
keeps j <= i + delta; window_left = W >= 0 also keeps only j >= i + delta - W.
"""
import numpy as np
import pytest
import torch

import oracle


def _mask(s_q, s_kv, mask, window):
    delta = s_kv - s_q if mask == "bottom_right" else 0
    i = np.arange(s_q)[:, None]
    j = np.arange(s_kv)[None, :]
    ok = np.ones((s_q, s_kv), bool)
    if mask != "none":
        ok &= j <= i + delta
    if window >= 0:
        ok &= j >= i + delta - window
    return ok


def _rand(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float64)


def _torch_ref(q, k, v, do, scale, mask, window):
    """float64 torch SDPA with a boolean mask and repeated K/V heads."""
    b, h, s_q, d = q.shape
    h_kv, s_kv = k.shape[1], k.shape[2]
    g = h // h_kv
    ok = torch.from_numpy(_mask(s_q, s_kv, mask, window))
    live = ok.any(dim=1)
    qq, kk, vv = (x.clone().requires_grad_(True) for x in (q, k, v))
    kr, vr = kk.repeat_interleave(g, dim=1), vv.repeat_interleave(g, dim=1)
    # rows without a visible key are NaN in torch; give them one fake key and
    # zero them afterwards (the definition makes them O = 0, no gradient)
    ok_safe = ok.clone()
    ok_safe[~live, 0] = True
    o = torch.nn.functional.scaled_dot_product_attention(qq, kr, vr, attn_mask=ok_safe,
                                                         scale=scale)
    o = o * live[None, None, :, None]
    (o * do).sum().backward()
    s = torch.einsum("bhid,bhjd->bhij", q, k.repeat_interleave(g, dim=1)) * scale
    s = s.masked_fill(~ok, float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    return o.detach(), lse, qq.grad, kk.grad, vv.grad, live


CASES = [
    # b, h, h_kv, s_q, s_kv, d, mask, window
    (1, 2, 2, 9, 9, 4, "bottom_right", -1),
    (2, 4, 2, 7, 12, 8, "bottom_right", -1),
    (1, 3, 1, 12, 7, 4, "bottom_right", -1),   # s_q > s_kv: leading dead rows
    (1, 2, 1, 10, 10, 4, "top_left", 3),
    (2, 4, 1, 8, 13, 4, "bottom_right", 2),
    (1, 2, 2, 11, 6, 8, "none", 2),
    (1, 6, 3, 16, 16, 8, "top_left", -1),
    (1, 4, 4, 5, 9, 4, "top_left", 0),
]


@pytest.mark.parametrize("case", CASES)
def test_extended_oracle_matches_torch_float64(case):
    b, h, h_kv, s_q, s_kv, d, mask, window = case
    seed = 700 + CASES.index(case)
    q, k, v = _rand((b, h, s_q, d), seed), _rand((b, h_kv, s_kv, d), seed + 1), \
        _rand((b, h_kv, s_kv, d), seed + 2)
    do = _rand((b, h, s_q, d), seed + 3)
    scale = 0.37
    o, lse = oracle.sdpa_fwd_ex(q, k, v, scale, mask, window)
    dq, dk, dv = oracle.sdpa_bwd_ex(q, k, v, do, scale, mask, window)
    ro, rlse, rdq, rdk, rdv, live = _torch_ref(q, k, v, do, scale, mask, window)
    np.testing.assert_allclose(o, ro.numpy(), rtol=0, atol=1e-12)
    live = live.numpy()
    np.testing.assert_allclose(lse[..., live], rlse.numpy()[..., live], rtol=0, atol=1e-12)
    assert np.all(np.isneginf(lse[..., ~live]))
    np.testing.assert_allclose(dq, rdq.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk, rdk.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dv, rdv.numpy(), rtol=0, atol=1e-11)


def _numpy_brute(q, k, v, scale, ok):
    """Full-matrix softmax of one problem, written independently."""
    s = scale * q @ k.T
    s = np.where(ok, s, -np.inf)
    out = np.zeros((q.shape[0], v.shape[1]))
    lse = np.full(q.shape[0], -np.inf)
    for i in range(q.shape[0]):
        if not ok[i].any():
            continue
        m = s[i][ok[i]].max()
        e = np.where(ok[i], np.exp(s[i] - m), 0.0)
        out[i] = e @ v / e.sum()
        lse[i] = m + np.log(e.sum())
    return out, lse


@pytest.mark.parametrize("mask,window", [("bottom_right", -1), ("bottom_right", 1),
                                         ("top_left", 2), ("none", 0)])
def test_extended_oracle_brute_force(mask, window):
    rng = np.random.default_rng(5)
    for s_q, s_kv in ((6, 6), (4, 9), (9, 4)):
        q, k, v = rng.normal(size=(s_q, 3)), rng.normal(size=(s_kv, 3)), rng.normal(size=(s_kv, 3))
        o, lse = oracle.attn_fwd_rows_ex(q, k, v, np.arange(s_q), 0.8, mask, window)
        ro, rlse = _numpy_brute(q, k, v, 0.8, _mask(s_q, s_kv, mask, window))
        np.testing.assert_allclose(o, ro, rtol=0, atol=1e-13)
        assert np.array_equal(np.isneginf(lse), np.isneginf(rlse))
        fin = np.isfinite(rlse)
        np.testing.assert_allclose(lse[fin], rlse[fin], rtol=0, atol=1e-13)


@pytest.mark.parametrize("mask", ["top_left", "bottom_right"])
def test_zero_window_closed_form(mask):
    # causal + window 0: row i sees exactly key i + delta (when it exists)
    s_q, s_kv, d = 6, 9, 4
    q, k, v = _rand((1, 1, s_q, d), 1), _rand((1, 1, s_kv, d), 2), _rand((1, 1, s_kv, d), 3)
    o, lse = oracle.sdpa_fwd_ex(q, k, v, 0.5, mask, 0)
    delta = s_kv - s_q if mask == "bottom_right" else 0
    for i in range(s_q):
        j = i + delta
        np.testing.assert_allclose(o[0, 0, i], v[0, 0, j].numpy(), rtol=0, atol=1e-15)
        assert abs(lse[0, 0, i] - 0.5 * float(q[0, 0, i] @ k[0, 0, j])) < 1e-14


def test_bottom_right_dead_rows_and_gradients():
    s_q, s_kv, d = 8, 5, 4
    q, k, v = _rand((1, 1, s_q, d), 11), _rand((1, 1, s_kv, d), 12), _rand((1, 1, s_kv, d), 13)
    do = _rand((1, 1, s_q, d), 14)
    o, lse = oracle.sdpa_fwd_ex(q, k, v, 0.5, "bottom_right")
    dead = s_q - s_kv  # rows i < s_q - s_kv see no key
    assert np.all(o[0, 0, :dead] == 0) and np.all(np.isneginf(lse[0, 0, :dead]))
    assert np.all(np.isfinite(lse[0, 0, dead:]))
    dq, dk, dv = oracle.sdpa_bwd_ex(q, k, v, do, 0.5, "bottom_right")
    assert np.all(dq[0, 0, :dead] == 0)
    # the last row sees every key: it equals the unmasked attention of that row
    full_o, _ = oracle.sdpa_fwd_ex(q, k, v, 0.5, "none")
    np.testing.assert_allclose(o[0, 0, -1], full_o[0, 0, -1], rtol=0, atol=1e-15)


def test_reductions_to_the_plain_cases():
    q, k, v = _rand((2, 4, 10, 8), 21), _rand((2, 4, 10, 8), 22), _rand((2, 4, 10, 8), 23)
    do = _rand((2, 4, 10, 8), 24)
    base = oracle.sdpa_fwd(q, k, v, 0.3, True)
    for mask, window in (("bottom_right", -1), ("top_left", 10), ("top_left", 25)):
        got = oracle.sdpa_fwd_ex(q, k, v, 0.3, mask, window)
        np.testing.assert_array_equal(got[0], base[0])
        np.testing.assert_array_equal(got[1], base[1])
    gb = oracle.sdpa_bwd(q, k, v, do, 0.3, True)
    ge = oracle.sdpa_bwd_ex(q, k, v, do, 0.3, "bottom_right", -1)
    for a, b in zip(ge, gb):
        np.testing.assert_array_equal(a, b)


def test_gqa_is_mha_on_repeated_heads_with_group_summed_grads():
    b, h, h_kv, s, d = 2, 6, 2, 9, 4
    g = h // h_kv
    q, k, v, do = _rand((b, h, s, d), 31), _rand((b, h_kv, s, d), 32), \
        _rand((b, h_kv, s, d), 33), _rand((b, h, s, d), 34)
    kr, vr = k.repeat_interleave(g, dim=1), v.repeat_interleave(g, dim=1)
    for mask, window in (("top_left", -1), ("bottom_right", 3), ("none", -1)):
        o, lse = oracle.sdpa_fwd_ex(q, k, v, 0.4, mask, window)
        ro, rlse = oracle.sdpa_fwd_ex(q, kr, vr, 0.4, mask, window)
        np.testing.assert_array_equal(o, ro)
        np.testing.assert_array_equal(lse, rlse)
        dq, dk, dv = oracle.sdpa_bwd_ex(q, k, v, do, 0.4, mask, window)
        rdq, rdk, rdv = oracle.sdpa_bwd_ex(q, kr, vr, do, 0.4, mask, window)
        np.testing.assert_array_equal(dq, rdq)
        np.testing.assert_allclose(dk, rdk.reshape(b, h_kv, g, s, d).sum(2), rtol=0, atol=1e-13)
        np.testing.assert_allclose(dv, rdv.reshape(b, h_kv, g, s, d).sum(2), rtol=0, atol=1e-13)


@pytest.mark.parametrize("mask,window", [("bottom_right", 1), ("top_left", 2)])
def test_extended_grads_by_finite_differences(mask, window):
    b, h, h_kv, s_q, s_kv, d = 1, 2, 1, 5, 7, 3
    q, k, v, do = _rand((b, h, s_q, d), 41), _rand((b, h_kv, s_kv, d), 42), \
        _rand((b, h_kv, s_kv, d), 43), _rand((b, h, s_q, d), 44)
    q, k, v, do = (x.numpy() for x in (q, k, v, do))
    dq, dk, dv = oracle.sdpa_bwd_ex(q, k, v, do, 0.6, mask, window)

    def loss(qq, kk, vv):
        return float((oracle.sdpa_fwd_ex(qq, kk, vv, 0.6, mask, window)[0] * do).sum())

    eps = 1e-6
    for name, x, gx in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args = {"q": q, "k": k, "v": v}
            args[name] = xp
            lp = loss(args["q"], args["k"], args["v"])
            args[name] = xm
            lm = loss(args["q"], args["k"], args["v"])
            num[idx] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(gx, num, rtol=1e-6, atol=1e-8, err_msg=name)


def test_extended_varlen_equals_dense_per_sequence():
    h, h_kv, d = 4, 2, 8
    lq, lk = [5, 0, 9, 3], [7, 4, 9, 0]
    cu_q = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    q, k, v = _rand((cu_q[-1], h, d), 51), _rand((cu_k[-1], h_kv, d), 52), \
        _rand((cu_k[-1], h_kv, d), 53)
    do = _rand((cu_q[-1], h, d), 54)
    for mask, window in (("bottom_right", -1), ("top_left", 2), ("bottom_right", 1)):
        o, lse = oracle.sdpa_varlen_fwd_ex(q, k, v, cu_q, cu_k, 0.5, mask, window)
        dq, dk, dv = oracle.sdpa_varlen_bwd_ex(q, k, v, do, cu_q, cu_k, 0.5, mask, window)
        for n in range(len(lq)):
            qs, ks = slice(cu_q[n], cu_q[n + 1]), slice(cu_k[n], cu_k[n + 1])
            if lq[n] == 0:
                continue
            qd = q[qs].permute(1, 0, 2)[None]
            kd, vd = k[ks].permute(1, 0, 2)[None], v[ks].permute(1, 0, 2)[None]
            dod = do[qs].permute(1, 0, 2)[None]
            ro, rlse = oracle.sdpa_fwd_ex(qd, kd, vd, 0.5, mask, window)
            np.testing.assert_array_equal(o[qs], ro[0].transpose(1, 0, 2))
            np.testing.assert_array_equal(lse[qs], rlse[0].T)
            if lk[n] == 0:
                continue
            rdq, rdk, rdv = oracle.sdpa_bwd_ex(qd, kd, vd, dod, 0.5, mask, window)
            np.testing.assert_allclose(dq[qs], rdq[0].transpose(1, 0, 2), rtol=0, atol=1e-14)
            np.testing.assert_allclose(dk[ks], rdk[0].transpose(1, 0, 2), rtol=0, atol=1e-14)
            np.testing.assert_allclose(dv[ks], rdv[0].transpose(1, 0, 2), rtol=0, atol=1e-14)


ROW_CASES = [
    # s_q, s_kv, mask, window, h, h_kv
    (9, 13, "bottom_right", 2, 4, 2),    # s_q < s_kv, window, GQA groups of 2
    (13, 9, "bottom_right", -1, 2, 1),   # s_q > s_kv: leading dead rows, MQA
    (11, 11, "top_left", 3, 6, 3),
    (10, 7, "none", 1, 2, 2),
]


@pytest.mark.parametrize("case", ROW_CASES)
def test_row_sampled_extended_entry_points_match_full(case):
    """The row-selecting calls that check full-size GPU results (one query
    head and its key/value head at a time, rows listed in any order) equal
    the matching rows of the full extended calls, and those rows equal
    torch's float64 reference; dK/dV of a key/value head are the sums of its
    group's per-query-head row results."""
    s_q, s_kv, mask, window, h, h_kv = case
    d, scale, g = 4, 0.45, h // h_kv
    seed = 800 + ROW_CASES.index(case)
    q, k, v = _rand((1, h, s_q, d), seed), _rand((1, h_kv, s_kv, d), seed + 1), \
        _rand((1, h_kv, s_kv, d), seed + 2)
    do = _rand((1, h, s_q, d), seed + 3)
    o, lse = oracle.sdpa_fwd_ex(q, k, v, scale, mask, window)
    dq, dk, dv = oracle.sdpa_bwd_ex(q, k, v, do, scale, mask, window)
    ro, rlse, rdq, rdk, rdv, live = _torch_ref(q, k, v, do, scale, mask, window)
    rng = np.random.default_rng(seed)
    q_rows = rng.permutation(s_q)[: max(2, s_q - 3)].astype(np.int32)
    kv_rows = rng.permutation(s_kv)[: max(2, s_kv - 2)].astype(np.int32)
    for hk in range(h_kv):
        sum_dk = sum_dv = 0
        for hq in range(hk * g, (hk + 1) * g):
            args = (q[0, hq], k[0, hk], v[0, hk])
            fo, flse = oracle.attn_fwd_rows_ex(*args, q_rows, scale, mask, window)
            np.testing.assert_array_equal(fo, o[0, hq][q_rows])
            np.testing.assert_array_equal(flse, lse[0, hq][q_rows])
            np.testing.assert_allclose(fo, ro[0, hq][q_rows].numpy(), rtol=0, atol=1e-12)
            bq, bk, bv = oracle.attn_bwd_rows_ex(*args, do[0, hq], q_rows, kv_rows, scale, mask,
                                                 window)
            np.testing.assert_array_equal(bq, dq[0, hq][q_rows])
            np.testing.assert_allclose(bq, rdq[0, hq][q_rows].numpy(), rtol=0, atol=1e-11)
            sum_dk, sum_dv = sum_dk + bk, sum_dv + bv
        np.testing.assert_allclose(sum_dk, dk[0, hk][kv_rows], rtol=0, atol=1e-13)
        np.testing.assert_allclose(sum_dv, dv[0, hk][kv_rows], rtol=0, atol=1e-13)
        np.testing.assert_allclose(sum_dk, rdk[0, hk][kv_rows].numpy(), rtol=0, atol=1e-11)
        np.testing.assert_allclose(sum_dv, rdv[0, hk][kv_rows].numpy(), rtol=0, atol=1e-11)
    if mask == "bottom_right" and s_q > s_kv:  # the listed rows include dead ones
        assert (~live.numpy())[q_rows].any()


# ------------------------------------------------------------------ FP8 E4M3
def test_e4m3_decoder_matches_torch_on_every_code():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_decode(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2  # S.1111.111
    np.testing.assert_array_equal(got[~nan], ref[~nan])


def test_e4m3_decoder_values_from_the_format():
    # 1.0 = 0.0111.000, 448 = 0.1111.110, smallest subnormal 2^-9 = 0.0000.001
    assert oracle.e4m3_decode(0x38) == 1.0
    assert oracle.e4m3_decode(0x7E) == 448.0
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9
    assert oracle.e4m3_decode(0xB8) == -1.0
    arr = oracle.e4m3_to_f64(np.array([0x38, 0x40, 0x08], np.uint8), 0.5)
    np.testing.assert_array_equal(arr, [0.5, 1.0, 0.5 * 2.0 ** -6])


def test_fp8_forward_is_attention_of_the_dequantized_values():
    g = torch.Generator().manual_seed(9)
    q, k, v = (torch.randn(1, 2, 20, 16, generator=g) for _ in range(3))
    enc = [x.mul(8.0).to(torch.float8_e4m3fn) for x in (q, k, v)]
    codes = [e.view(torch.uint8) for e in enc]
    real = [e.to(torch.float64) / 8.0 for e in enc]
    o, lse = oracle.sdpa_fwd_fp8(*codes, 0.125, 0.125, 0.125, 0.25, "bottom_right", 5)
    ro, rlse = oracle.sdpa_fwd_ex(*real, 0.25, "bottom_right", 5)
    np.testing.assert_array_equal(o, ro)
    np.testing.assert_array_equal(lse, rlse)
