"""Parity of the extended entry points (grouped key/value heads, bottom-right
causal alignment, left windows) against the fp64 oracle's extended
definitions, through the C ABI, on both forward kernels, dense and packed,
forward and backward.

Masks (cudnn-frontend PR #554 `sdpa` op: is_causal, causal_bottom_right,
window_left): query i sees key j iff lo_i <= j < hi_i, delta = Lkv - Lq for
bottom-right, hi_i = min(Lkv, i + delta + 1) when causal, lo_i = i + delta -
window_left when window_left >= 0.  Tolerances as in helpers.py.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import sdpa_inputs
from helpers import GRAD_TOL, O_TOL, check_lse, check_rel

pytestmark = pytest.mark.gpu

MASK_CODE = {"none": 0, "top_left": 1, "bottom_right": 2}


@pytest.fixture(scope="module")
def sdpa():
    import scaled_dot_product_04_gb300 as m
    m.load()
    return m


@pytest.fixture(params=[1, 2], ids=["one_tile", "two_tile"])
def variant(request, sdpa):
    sdpa.sdpa_set_forward_variant(request.param)
    yield request.param
    sdpa.sdpa_set_forward_variant(0)


def _grads_ok(got, ref, names=("dq", "dk", "dv")):
    for name, g, r in zip(names, got, ref):
        r = np.asarray(r)
        if np.abs(r).max() == 0:
            assert float(g.abs().max()) <= 1e-4, name
        else:
            check_rel(g, r, GRAD_TOL, name)


DENSE_CASES = [
    # b, h, h_kv, s_q, s_kv, d, mask, window
    (2, 8, 2, 300, 300, 128, "top_left", -1),          # GQA, group 4
    (1, 6, 1, 257, 515, 64, "top_left", -1),           # MQA
    (1, 4, 4, 200, 460, 128, "bottom_right", -1),      # s_q < s_kv
    (1, 4, 2, 460, 200, 64, "bottom_right", -1),       # s_q > s_kv: 260 dead rows
    (2, 4, 4, 600, 600, 128, "top_left", 0),           # one key per row
    (1, 4, 2, 700, 700, 128, "top_left", 150),         # window spanning tiles
    (1, 4, 4, 333, 777, 64, "bottom_right", 200),
    (1, 2, 1, 520, 400, 128, "none", 70),              # left bound only
    (1, 8, 2, 2100, 2100, 128, "bottom_right", -1),    # long enough for the two-tile choice
    (1, 4, 2, 640, 900, 128, "bottom_right", 300),     # band of a bottom-right window, GQA
    (1, 4, 2, 900, 350, 128, "bottom_right", 100),     # s_q > s_kv: keyless leading tiles
]


@pytest.mark.parametrize("case", DENSE_CASES, ids=lambda c: f"b{c[0]}h{c[1]}kv{c[2]}s{c[3]}x{c[4]}d{c[5]}_{c[6]}_w{c[7]}")
def test_ext_dense_fwd(sdpa, variant, case):
    b, h, h_kv, s_q, s_kv, d, mask, window = case
    q, k, v, _ = sdpa_inputs.dense(b, h, s_q, s_kv, d, seed=3000 + s_q + s_kv, h_kv=h_kv)
    scale = 1.0 / math.sqrt(d)
    o, lse = sdpa.attention(q.cuda(), k.cuda(), v.cuda(), scale=scale, mask=mask,
                            window_left=window)
    torch.cuda.synchronize()
    ro, rlse = oracle.sdpa_fwd_ex(q, k, v, scale, mask, window)
    check_rel(o, ro, O_TOL[torch.bfloat16], "o")
    check_lse(lse, rlse)


@pytest.mark.usefixtures("bwd_variant")
@pytest.mark.parametrize("case", DENSE_CASES, ids=lambda c: f"b{c[0]}h{c[1]}kv{c[2]}s{c[3]}x{c[4]}d{c[5]}_{c[6]}_w{c[7]}")
def test_ext_dense_bwd(sdpa, case):
    b, h, h_kv, s_q, s_kv, d, mask, window = case
    q, k, v, do = sdpa_inputs.dense(b, h, s_q, s_kv, d, seed=4000 + s_q + s_kv, h_kv=h_kv)
    scale = 1.0 / math.sqrt(d)
    qc, kc, vc, doc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = sdpa.attention(qc, kc, vc, scale=scale, mask=mask, window_left=window)
    got = sdpa.attention_bwd(qc, kc, vc, o, doc, lse, scale=scale, mask=mask, window_left=window)
    torch.cuda.synchronize()
    assert got[1].shape == k.shape and got[2].shape == v.shape
    _grads_ok(got, oracle.sdpa_bwd_ex(q, k, v, do, scale, mask, window))


PACKED_CASES = [
    # lengths_q, lengths_kv, h, h_kv, d, mask, window
    ([130, 7, 300, 64], [130, 7, 300, 64], 4, 2, 128, "top_left", -1),
    ([100, 50, 260, 1], [180, 50, 130, 9], 4, 4, 64, "bottom_right", -1),
    ([90, 0, 400], [60, 33, 120], 2, 1, 128, "bottom_right", -1),   # s_q > s_kv in one
    ([300, 129, 257], [300, 129, 257], 6, 3, 128, "top_left", 100),
    ([200, 513], [450, 300], 4, 2, 64, "bottom_right", 64),
    ([70, 260], [0, 260], 2, 2, 128, "top_left", 5),                 # a sequence without keys
    ([520, 333], [700, 333], 4, 4, 128, "bottom_right", 150),
]


def _packed_run(sdpa, case, seed, backward):
    lq, lk, h, h_kv, d, mask, window = case
    q, k, v, do, cu_q, cu_kv = sdpa_inputs.packed(lq, lk, h, d, seed=seed, h_kv=h_kv)
    scale = 1.0 / math.sqrt(d)
    qc, kc, vc, doc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    cq, ck = cu_q.cuda(), cu_kv.cuda()
    o, lse = sdpa.attention_varlen(qc, kc, vc, cq, ck, max(lq), max(lk), scale=scale, mask=mask,
                                   window_left=window)
    got = None
    if backward:
        got = sdpa.attention_varlen_bwd(qc, kc, vc, o, doc, lse, cq, ck, max(lq), max(lk),
                                        scale=scale, mask=mask, window_left=window)
    torch.cuda.synchronize()
    return (q, k, v, do, cu_q, cu_kv, scale), o, lse, got


@pytest.mark.parametrize("case", PACKED_CASES, ids=lambda c: f"n{len(c[0])}h{c[2]}kv{c[3]}d{c[4]}_{c[5]}_w{c[6]}")
def test_ext_packed_fwd(sdpa, variant, case):
    lq, lk, h, h_kv, d, mask, window = case
    (q, k, v, _, cu_q, cu_kv, scale), o, lse, _ = _packed_run(sdpa, case, 5000 + sum(lq), False)
    ro, rlse = oracle.sdpa_varlen_fwd_ex(q, k, v, cu_q, cu_kv, scale, mask, window)
    check_rel(o, ro, O_TOL[torch.bfloat16], "o")
    check_lse(lse, rlse)
    for n in range(len(lq)):  # per sequence too
        s = slice(int(cu_q[n]), int(cu_q[n + 1]))
        if lq[n]:
            check_rel(o[s], ro[s], O_TOL[torch.bfloat16], f"o seq {n}")


@pytest.mark.usefixtures("bwd_variant")
@pytest.mark.parametrize("case", PACKED_CASES, ids=lambda c: f"n{len(c[0])}h{c[2]}kv{c[3]}d{c[4]}_{c[5]}_w{c[6]}")
def test_ext_packed_bwd(sdpa, case):
    lq, lk, h, h_kv, d, mask, window = case
    (q, k, v, do, cu_q, cu_kv, scale), _, _, got = _packed_run(sdpa, case, 6000 + sum(lq), True)
    ref = oracle.sdpa_varlen_bwd_ex(q, k, v, do, cu_q, cu_kv, scale, mask, window)
    assert got[1].shape == k.shape
    _grads_ok(got, ref)


@pytest.mark.usefixtures("bwd_variant")
def test_ext_fp16_gqa_window(sdpa, variant):
    b, h, h_kv, s, d = 1, 4, 2, 500, 128
    q, k, v, do = sdpa_inputs.dense(b, h, s, s, d, seed=77, dtype=torch.float16, h_kv=h_kv)
    scale = 1.0 / math.sqrt(d)
    qc, kc, vc, doc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = sdpa.attention(qc, kc, vc, scale=scale, mask="bottom_right", window_left=90)
    got = sdpa.attention_bwd(qc, kc, vc, o, doc, lse, scale=scale, mask="bottom_right",
                             window_left=90)
    torch.cuda.synchronize()
    ro, rlse = oracle.sdpa_fwd_ex(q, k, v, scale, "bottom_right", 90)
    check_rel(o, ro, O_TOL[torch.float16], "o")
    check_lse(lse, rlse)
    _grads_ok(got, oracle.sdpa_bwd_ex(q, k, v, do, scale, "bottom_right", 90))


def test_ext_plain_arguments_match_the_plain_calls(sdpa):
    # h_kv = h, mask = causal, no window through the _ex entry points gives
    # the plain calls' results bit for bit (same kernels, same schedule)
    b, h, s, d = 1, 4, 700, 128
    q, k, v, do = (x.cuda() for x in sdpa_inputs.dense(b, h, s, s, d, seed=5))
    scale = 1.0 / math.sqrt(d)
    o1, l1 = sdpa.attention(q, k, v, scale=scale, causal=True)
    o2, l2 = torch.empty_like(q), torch.empty_like(l1)
    sdpa.sdpa_fwd_ex(q, k, v, o2, l2, b, h, h, s, s, d, scale, 1, -1, 0)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    g1 = sdpa.attention_bwd(q, k, v, o1, do, l1, scale=scale, causal=True)
    ws = torch.empty(sdpa.sdpa_bwd_ex_workspace_size(b, h, s, d, 0), dtype=torch.uint8,
                     device="cuda")
    g2 = tuple(torch.empty_like(x) for x in (q, k, v))
    sdpa.sdpa_bwd_ex(q, k, v, o1, do, l1, *g2, b, h, h, s, s, d, scale, 1, -1, 0, 0, ws,
                     ws.numel())
    torch.cuda.synchronize()
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])  # dK, dV deterministic
    check_rel(g2[0], g1[0].double().cpu().numpy(), 1e-3, "dq")


def test_ext_validation(sdpa):
    from scaled_dot_product_04_gb300 import _lib as L
    q = torch.empty(1, 6, 128, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.empty(1, 4, 128, 64, dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(1, 6, 128, device="cuda")
    with pytest.raises(sdpa.SdpaError) as e:  # 6 is not a multiple of 4
        sdpa.sdpa_fwd_ex(q, k, k, o, lse, 1, 6, 4, 128, 128, 64, 0.1, 1, -1, 0)
    assert e.value.status == L.SDPA_ERR_INVALID_ARG and "multiple" in str(e.value)
    with pytest.raises(sdpa.SdpaError) as e:
        sdpa.sdpa_fwd_ex(q, k, k, o, lse, 1, 6, 3, 128, 128, 64, 0.1, 3, -1, 0)
    assert e.value.status == L.SDPA_ERR_INVALID_ARG and "mask" in str(e.value)
    with pytest.raises(sdpa.SdpaError) as e:
        sdpa.sdpa_fwd_ex(q, k, k, o, lse, 1, 6, 3, 128, 128, 64, 0.1, 1, -2, 0)
    assert e.value.status == L.SDPA_ERR_INVALID_ARG and "window" in str(e.value)


# ------------------------------------------------------------ deterministic backward
DET_DENSE = [
    (2, 4, 4, 333, 333, 128, "top_left", -1),
    (1, 8, 2, 700, 700, 64, "bottom_right", -1),
    (1, 4, 1, 300, 520, 128, "none", -1),
    (1, 4, 2, 640, 640, 128, "top_left", 100),
    (1, 2, 2, 460, 200, 128, "bottom_right", -1),   # dead rows
]


@pytest.mark.usefixtures("bwd_variant")
@pytest.mark.parametrize("case", DET_DENSE, ids=lambda c: f"b{c[0]}h{c[1]}kv{c[2]}s{c[3]}x{c[4]}d{c[5]}_{c[6]}_w{c[7]}")
def test_deterministic_dense_bwd_parity_and_bits(sdpa, case):
    b, h, h_kv, s_q, s_kv, d, mask, window = case
    q, k, v, do = sdpa_inputs.dense(b, h, s_q, s_kv, d, seed=7000 + s_q + s_kv, h_kv=h_kv)
    scale = 1.0 / math.sqrt(d)
    qc, kc, vc, doc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = sdpa.attention(qc, kc, vc, scale=scale, mask=mask, window_left=window)
    runs = [sdpa.attention_bwd(qc, kc, vc, o, doc, lse, scale=scale, mask=mask,
                               window_left=window, deterministic=True) for _ in range(3)]
    torch.cuda.synchronize()
    for name, i in (("dq", 0), ("dk", 1), ("dv", 2)):
        assert torch.equal(runs[0][i], runs[1][i]) and torch.equal(runs[0][i], runs[2][i]), name
    _grads_ok(runs[0], oracle.sdpa_bwd_ex(q, k, v, do, scale, mask, window))
    # dK, dV are the default path's bits; dQ agrees to rounding
    plain = sdpa.attention_bwd(qc, kc, vc, o, doc, lse, scale=scale, mask=mask, window_left=window)
    torch.cuda.synchronize()
    assert torch.equal(plain[1], runs[0][1]) and torch.equal(plain[2], runs[0][2])
    check_rel(runs[0][0], plain[0].double().cpu().numpy(), 1e-2, "dq vs default")


@pytest.mark.usefixtures("bwd_variant")
@pytest.mark.parametrize("case", PACKED_CASES[:4], ids=lambda c: f"n{len(c[0])}h{c[2]}kv{c[3]}d{c[4]}_{c[5]}_w{c[6]}")
def test_deterministic_packed_bwd(sdpa, case):
    lq, lk, h, h_kv, d, mask, window = case
    q, k, v, do, cu_q, cu_kv = sdpa_inputs.packed(lq, lk, h, d, seed=8000 + sum(lq), h_kv=h_kv)
    scale = 1.0 / math.sqrt(d)
    qc, kc, vc, doc, cq, ck = q.cuda(), k.cuda(), v.cuda(), do.cuda(), cu_q.cuda(), cu_kv.cuda()
    o, lse = sdpa.attention_varlen(qc, kc, vc, cq, ck, max(lq), max(lk), scale=scale, mask=mask,
                                   window_left=window)
    runs = [sdpa.attention_varlen_bwd(qc, kc, vc, o, doc, lse, cq, ck, max(lq), max(lk),
                                      scale=scale, mask=mask, window_left=window,
                                      deterministic=True) for _ in range(2)]
    torch.cuda.synchronize()
    for i in range(3):
        assert torch.equal(runs[0][i], runs[1][i])
    _grads_ok(runs[0], oracle.sdpa_varlen_bwd_ex(q, k, v, do, cu_q, cu_kv, scale, mask, window))


@pytest.mark.usefixtures("bwd_variant")
def test_deterministic_packed_bwd_without_keys_or_with_unseen_key_tiles(sdpa):
    """The deterministic dQ pass starts while the main kernel runs and reads
    the preprocess kernel's row terms without waiting itself: here every main
    CTA either has no key tile (no sequence has keys: the pass then follows
    the preprocess kernel in plain order) or sees no query for some of its key
    tiles (a bottom-right band of 6 keys leaves the first key tiles unseen)."""
    h, d = 2, 64
    lq, lk = [40, 7, 130], [0, 0, 0]
    q, k, v, do, cu_q, cu_kv = sdpa_inputs.packed(lq, lk, h, d, seed=8100)
    qc, doc, cq, ck = q.cuda(), do.cuda(), cu_q.cuda(), cu_kv.cuda()
    kc = torch.empty((8, h, d), dtype=q.dtype, device="cuda")  # capacity only, total_kv = 0
    o, lse = sdpa.attention_varlen(qc, kc, kc, cq, ck, max(lq), 0, scale=0.125, causal=True,
                                   total_kv=0)
    dq, dk, dv = sdpa.attention_varlen_bwd(qc, kc, kc, o, doc, lse, cq, ck, max(lq), 0,
                                           scale=0.125, causal=True, deterministic=True,
                                           total_kv=0)
    torch.cuda.synchronize()
    assert torch.isneginf(lse).all() and float(o.abs().max()) == 0.0
    assert float(dq.abs().max()) == 0.0
    lq, lk = [50, 200, 64], [400, 390, 500]
    q, k, v, do, cu_q, cu_kv = sdpa_inputs.packed(lq, lk, h, d, seed=8101)
    qc, kc, vc, doc, cq, ck = q.cuda(), k.cuda(), v.cuda(), do.cuda(), cu_q.cuda(), cu_kv.cuda()
    o, lse = sdpa.attention_varlen(qc, kc, vc, cq, ck, max(lq), max(lk), scale=0.125,
                                   mask="bottom_right", window_left=5)
    runs = [sdpa.attention_varlen_bwd(qc, kc, vc, o, doc, lse, cq, ck, max(lq), max(lk),
                                      scale=0.125, mask="bottom_right", window_left=5,
                                      deterministic=True) for _ in range(2)]
    torch.cuda.synchronize()
    for i in range(3):
        assert torch.equal(runs[0][i], runs[1][i])
    _grads_ok(runs[0], oracle.sdpa_varlen_bwd_ex(q, k, v, do, cu_q, cu_kv, 0.125, "bottom_right", 5))


def test_deterministic_workspace_is_the_row_terms(sdpa):
    assert sdpa.sdpa_bwd_ex_workspace_size(2, 3, 100, 128, 1) == 2 * 3 * 100 * 16 + 256 - (2 * 3 * 100 * 16) % 256
    assert sdpa.sdpa_bwd_ex_workspace_size(2, 3, 100, 128, 0) == sdpa.sdpa_bwd_workspace_size(2, 3, 100, 128)


def test_ext_fp16_packed_window(sdpa, variant):
    """fp16 packed with a left window on both forward kernels."""
    lens, h, h_kv, d = [333, 600, 90], 4, 2, 128
    q, k, v, do, cu, _ = sdpa_inputs.packed(lens, lens, h, d, seed=78, dtype=torch.float16,
                                           h_kv=h_kv)
    scale = 1.0 / math.sqrt(d)
    o, lse = sdpa.attention_varlen(q.cuda(), k.cuda(), v.cuda(), cu.cuda(), cu.cuda(), max(lens),
                                   max(lens), scale=scale, causal=True, window_left=130)
    torch.cuda.synchronize()
    ro, rlse = oracle.sdpa_varlen_fwd_ex(q, k, v, cu, cu, scale, "top_left", 130)
    check_rel(o, ro, O_TOL[torch.float16], "o")
    check_lse(lse, rlse)
