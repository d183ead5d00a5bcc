"""Forward parity: CUDA path (through the C ABI) vs the fp64 oracle.

Small and medium problems are compared element by element on every output
(the full-size workloads, whole slices at a time, are in
test_gpu_full_slices.py).  Edge cases: ragged tails, s_q != s_kv, several tiles,
dead rows (zero keys), THD with zero-length sequences, NaN-poisoned capacity
tails, fp16, determinism, and no host synchronisation.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import sdpa_inputs
from helpers import O_TOL, check_lse, check_rel, np64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sdpa():
    import scaled_dot_product_04_gb300 as m
    m.load()
    return m


@pytest.fixture(autouse=True, params=[1, 2], ids=["one_tile", "two_tile"])
def fwd_variant(request, sdpa):
    """Every forward case runs on both forward kernels (128- and 256-row units)."""
    sdpa.sdpa_set_forward_variant(request.param)
    yield request.param
    sdpa.sdpa_set_forward_variant(0)


def _dense_case(sdpa, b, h, s_q, s_kv, d, causal, dtype=torch.bfloat16, seed=0, qk_mult=1.0):
    q, k, v, _ = sdpa_inputs.dense(b, h, s_q, s_kv, d, seed=seed, dtype=dtype, qk_mult=qk_mult)
    scale = 1.0 / math.sqrt(d)
    o, lse = sdpa.attention(q.cuda(), k.cuda(), v.cuda(), scale=scale, causal=causal)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.sdpa_fwd(q, k, v, scale, causal)
    check_rel(o, o_ref, O_TOL[dtype], "O")
    check_lse(lse, lse_ref)
    return o, lse


def test_config1_full(sdpa):
    w = sdpa_inputs.WORKLOADS["c1_b1h2s128d64_causal"]
    _dense_case(sdpa, w.b, w.h, w.s, w.s, w.d, w.causal, seed=w.seed)


def test_config2_full(sdpa):
    w = sdpa_inputs.WORKLOADS["c2_b4h16s1024d64_causal"]
    _dense_case(sdpa, w.b, w.h, w.s, w.s, w.d, w.causal, seed=w.seed)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("s_q,s_kv", [(333, 333), (1, 1), (129, 129), (200, 461), (461, 200),
                                      (512, 512)])
def test_dense_shapes(sdpa, d, causal, s_q, s_kv):
    _dense_case(sdpa, 2, 3, s_q, s_kv, d, causal, seed=s_q * 7 + s_kv)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_dense_fp16(sdpa, d, causal):
    _dense_case(sdpa, 1, 4, 300, 300, d, causal, dtype=torch.float16, seed=77)


def test_sharpened_softmax(sdpa):
    """Q, K x 2 (the long-context recipe) at a size the oracle runs in full."""
    _dense_case(sdpa, 1, 4, 1000, 1000, 128, True, seed=1005, qk_mult=2.0)


def test_large_scores_rescale(sdpa):
    """Scores growing along the key axis force repeated rescales of O."""
    b, h, s, d = 1, 2, 640, 64
    g = torch.Generator().manual_seed(5)
    q = (torch.randn(b, h, s, d, generator=g) * 3).bfloat16()
    k = (torch.randn(b, h, s, d, generator=g) * torch.linspace(0.2, 4, s)[None, None, :, None]
         ).bfloat16()
    v = torch.randn(b, h, s, d, generator=g).bfloat16()
    for causal in (False, True):
        o, lse = sdpa.attention(q.cuda(), k.cuda(), v.cuda(), scale=0.125, causal=causal)
        o_ref, lse_ref = oracle.sdpa_fwd(q, k, v, 0.125, causal)
        check_rel(o, o_ref, O_TOL[torch.bfloat16], "O")
        check_lse(lse, lse_ref)


def test_zero_keys_dense(sdpa):
    q = torch.randn(1, 2, 130, 64).bfloat16().cuda()
    k = torch.empty(1, 2, 0, 64, dtype=torch.bfloat16, device="cuda")
    o, lse = sdpa.attention(q, k, k, scale=0.125, causal=True)
    torch.cuda.synchronize()
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


def test_lse_optional(sdpa):
    q, k, v, _ = sdpa_inputs.dense(1, 2, 256, 256, 64, seed=3)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    o = torch.empty_like(q)
    sdpa.sdpa_fwd(q, k, v, o, None, 1, 2, 256, 256, 64, 0.125, 1, 0)
    o2, _ = sdpa.attention(q, k, v, scale=0.125, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o, o2)


def test_deterministic_and_guarded(sdpa):
    """Bitwise-identical reruns; nothing written outside O and LSE."""
    b, h, s, d = 2, 4, 700, 128
    q, k, v, _ = sdpa_inputs.dense(b, h, s, s, d, seed=21)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    n = b * h * s * d
    guard = 4096
    o_buf = torch.full((n + 2 * guard,), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse_buf = torch.full((b * h * s + 2 * guard,), 12345.0, device="cuda")
    o = o_buf[guard:guard + n].view(b, h, s, d)
    lse = lse_buf[guard:guard + b * h * s].view(b, h, s)
    sdpa.sdpa_fwd(q, k, v, o, lse, b, h, s, s, d, 1 / math.sqrt(d), 1, 0)
    o_1, lse_1 = o.clone(), lse.clone()
    sdpa.sdpa_fwd(q, k, v, o, lse, b, h, s, s, d, 1 / math.sqrt(d), 1, 0)
    torch.cuda.synchronize()
    assert torch.equal(o, o_1) and torch.equal(lse, lse_1)
    assert torch.isnan(o_buf[:guard].float()).all() and torch.isnan(o_buf[-guard:].float()).all()
    assert (lse_buf[:guard] == 12345.0).all() and (lse_buf[-guard:] == 12345.0).all()


def test_no_host_sync(sdpa):
    q, k, v, _ = sdpa_inputs.dense(1, 2, 256, 256, 64, seed=4)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    o = torch.empty_like(q)
    lse = torch.empty(1, 2, 256, device="cuda")
    lens = [100, 0, 156]
    qv, kv, vv, _, cu, _ = sdpa_inputs.packed(lens, lens, 2, 64, seed=4)
    qv, kv, vv, cu = qv.cuda(), kv.cuda(), vv.cuda(), cu.cuda()
    ov, lsev = torch.empty_like(qv), torch.empty(256, 2, device="cuda")
    torch.cuda.synchronize()
    torch.cuda.set_sync_debug_mode("error")
    try:
        sdpa.sdpa_fwd(q, k, v, o, lse, 1, 2, 256, 256, 64, 0.125, 1, 0)
        sdpa.sdpa_varlen_fwd(qv, kv, vv, ov, lsev, cu, cu, 3, 256, 256, 156, 156, 2, 64, 0.125, 1,
                             0)
    finally:
        torch.cuda.set_sync_debug_mode("default")
    torch.cuda.synchronize()


# ------------------------------------------------------------------ packed
def _varlen_case(sdpa, lens_q, lens_kv, h, d, causal, dtype=torch.bfloat16, seed=0,
                 capacity_pad=0):
    q, k, v, _, cu_q, cu_kv = sdpa_inputs.packed(lens_q, lens_kv, h, d, seed=seed, dtype=dtype)
    tq, tkv = q.shape[0], k.shape[0]
    scale = 1.0 / math.sqrt(d)

    def on_gpu(x, pad):
        if pad == 0:
            return x.cuda()
        buf = torch.full((x.shape[0] + pad,) + tuple(x.shape[1:]), float("nan"), dtype=x.dtype,
                         device="cuda")
        buf[:x.shape[0]] = x.cuda()
        return buf

    qg, kg, vg = on_gpu(q, capacity_pad), on_gpu(k, capacity_pad), on_gpu(v, capacity_pad)
    o, lse = sdpa.attention_varlen(qg, kg, vg, cu_q.cuda(), cu_kv.cuda(), max(lens_q),
                                   max(max(lens_kv), 0), scale=scale, causal=causal, total_q=tq,
                                   total_kv=tkv)
    torch.cuda.synchronize()
    o, lse = o[:tq], lse[:tq]
    o_ref, lse_ref = oracle.sdpa_varlen_fwd(q, k, v, cu_q, cu_kv, scale, causal)
    check_rel(o, o_ref, O_TOL[dtype], "O")
    check_lse(lse, lse_ref)
    # per-sequence report (the pages check THD per sequence)
    for n in range(len(lens_q)):
        a, e = int(cu_q[n]), int(cu_q[n + 1])
        if e > a and np.abs(o_ref[a:e]).max() > 0:
            check_rel(o[a:e], o_ref[a:e], O_TOL[dtype], f"O seq {n}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_mixed(sdpa, d, causal):
    lens = [1, 127, 128, 129, 397, 0, 513, 64]
    _varlen_case(sdpa, lens, lens, 3, d, causal, seed=11)


def test_varlen_nan_capacity_tail(sdpa):
    """Three sequences totalling 397 tokens in NaN-tailed capacity buffers."""
    lens = [100, 200, 97]
    _varlen_case(sdpa, lens, lens, 4, 128, True, seed=12, capacity_pad=300)
    _varlen_case(sdpa, lens, lens, 4, 64, False, seed=13, capacity_pad=300)


def test_varlen_zero_length_kv(sdpa):
    """A sequence with queries but no keys: its rows are dead (O = 0, LSE = -inf)."""
    lens_q = [50, 70, 130]
    lens_kv = [50, 0, 200]
    _varlen_case(sdpa, lens_q, lens_kv, 2, 128, False, seed=14)
    _varlen_case(sdpa, lens_q, lens_kv, 2, 64, True, seed=15)


def test_varlen_fp16(sdpa):
    lens = [300, 17, 256]
    _varlen_case(sdpa, lens, lens, 2, 128, True, dtype=torch.float16, seed=16)


def test_varlen_single_equals_dense(sdpa):
    L, h, d = 777, 4, 128
    q, k, v, _ = sdpa_inputs.dense(1, h, L, L, d, seed=17)
    o_d, lse_d = sdpa.attention(q.cuda(), k.cuda(), v.cuda(), scale=0.1, causal=True)
    pk = lambda x: x[0].permute(1, 0, 2).contiguous().cuda()  # noqa: E731
    cu = torch.tensor([0, L], dtype=torch.int32, device="cuda")
    o_v, lse_v = sdpa.attention_varlen(pk(q), pk(k), pk(v), cu, cu, L, L, scale=0.1, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o_v.permute(1, 0, 2)[None], o_d)
    assert torch.equal(lse_v.T[None], lse_d)


def test_device_error_word_clean(sdpa):
    sdpa.sdpa_check_device_error()


def test_validation_on_gpu(sdpa):
    q = torch.randn(1, 1, 128, 64, device="cuda").bfloat16()
    o = torch.empty_like(q)
    flat = torch.empty(128 * 64 + 8, dtype=torch.bfloat16, device="cuda")
    mis = flat[1:1 + 128 * 64].view(1, 1, 128, 64)
    with pytest.raises(sdpa.SdpaError) as e:
        sdpa.sdpa_fwd(mis, q, q, o, None, 1, 1, 128, 128, 64, 0.125, 1, 0)
    assert e.value.status == 3
    with pytest.raises(sdpa.SdpaError) as e:
        sdpa.sdpa_fwd(q, q, q, q, None, 1, 1, 128, 128, 64, 0.125, 1, 0)
    assert e.value.status == 1
    with pytest.raises(sdpa.SdpaError) as e:
        sdpa.sdpa_fwd(q, q, q, o, None, 1, 1, 128, 128, 96, 0.125, 1, 0)
    assert e.value.status == 2


# ------------------------------------------------- many units per persistent CTA
@pytest.mark.parametrize("causal", [False, True])
def test_many_short_units_dense(sdpa, causal):
    """768+ query tiles with 1-3 key tiles each: every CTA runs many units back to back."""
    _dense_case(sdpa, 8, 32, 300, 300, 128, causal, seed=41)
    _dense_case(sdpa, 4, 48, 260, 260, 64, causal, seed=42)


def test_many_short_units_varlen_deterministic(sdpa):
    lens = [129, 300, 1, 256, 257, 64, 200, 130] * 6
    _varlen_case(sdpa, lens, lens, 16, 128, True, seed=43)
    q, k, v, _, cu, _ = sdpa_inputs.packed(lens, lens, 16, 128, seed=44)
    q, k, v, cu = q.cuda(), k.cuda(), v.cuda(), cu.cuda()
    a = sdpa.attention_varlen(q, k, v, cu, cu, max(lens), max(lens), scale=0.088, causal=True)
    b = sdpa.attention_varlen(q, k, v, cu, cu, max(lens), max(lens), scale=0.088, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("d,n", [(128, 90), (128, 120), (64, 300)])
def test_many_sequences_unit_orders(sdpa, d, n):
    """Packed unit lists of the one-tile forward: length-sorted sequence-major
    (sequence table cached in shared memory), sequence-major in the given order
    (over 256 sequences), and latest-tile-first over all slices (table not
    cached: more than 95 sequences at d = 128); with empty sequences."""
    g = np.random.default_rng(n)
    lens = g.integers(0, 300, n).tolist()
    lens[3] = 0
    lens[7] = 513
    _varlen_case(sdpa, lens, lens, 2, d, True, seed=45 + n)


# ------------------------------------- unit orders of problems larger than L2
# K + V above 64 MiB switch the one-tile forward to slice-group order (dense:
# batch by batch; packed: sequence by sequence, longest first when the
# sequence table fits in shared memory).  Sampled rows against the oracle.
def _sampled_rows(n, salt):
    return np.unique(np.array([0, n - 1, n // 2, (salt * 13) % n, (salt * 29 + 5) % n], np.int32))


def test_slice_major_dense_one_tile(sdpa):
    b, h, s, d = 8, 32, 1024, 128  # K + V = 134 MB
    q, k, v, _ = sdpa_inputs.dense(b, h, s, s, d, seed=61)
    sdpa.sdpa_set_forward_variant(1)
    try:
        o, lse = sdpa.attention(q.cuda(), k.cuda(), v.cuda(), scale=0.088, causal=True)
        torch.cuda.synchronize()
    finally:
        sdpa.sdpa_set_forward_variant(0)
    o, lse = o.cpu(), lse.cpu()
    for bb, hh in [(0, 0), (3, 17), (7, 31)]:
        rows = _sampled_rows(s, bb * 32 + hh)
        ro, rl = oracle.attn_fwd_rows(q[bb, hh], k[bb, hh], v[bb, hh], rows, 0.088, True)
        check_rel(o[bb, hh][rows], ro, O_TOL[torch.bfloat16], f"o[{bb},{hh}]")
        check_lse(lse[bb, hh][rows], rl)


@pytest.mark.parametrize("d,n,lo,hi", [(128, 40, 1, 400),     # sorted sequence-major
                                        (64, 300, 0, 60),      # sequence-major, given order
                                        (128, 120, 0, 120)])   # table not cached
def test_slice_major_packed_one_tile(sdpa, d, n, lo, hi):
    h = 32
    g = np.random.default_rng(n + d)
    lens = g.integers(lo, hi, n).tolist()
    lens[1] = 0
    lens[2] = hi + 200
    q, k, v, _, cu, _ = sdpa_inputs.packed(lens, lens, h, d, seed=62 + n)
    assert 2 * k.numel() * 2 > (64 << 20)
    o, lse = sdpa.attention_varlen(q.cuda(), k.cuda(), v.cuda(), cu.cuda(), cu.cuda(), max(lens),
                                   max(lens), scale=1.0 / math.sqrt(d), causal=True)
    torch.cuda.synchronize()
    o, lse = o.cpu(), lse.cpu()
    cl = cu.tolist()
    for i, L in enumerate(lens):
        if L == 0:
            continue
        hh = (i * 7) % h
        a, e = cl[i], cl[i + 1]
        rows = _sampled_rows(L, i)
        ro, rl = oracle.attn_fwd_rows(q[a:e, hh], k[a:e, hh], v[a:e, hh], rows, 1.0 / math.sqrt(d),
                                      True)
        check_rel(o[a:e, hh][rows], ro, O_TOL[torch.bfloat16], f"o seq {i}")
        check_lse(lse[a:e, hh][rows], rl, f"lse seq {i}")


def test_packed_kernel_choice(sdpa):
    """Packed lists that fit the two-tile kernel's sequence table (95 sequences
    at d = 128) run it by default, whatever their lengths; a longer list of
    short sequences runs the one-tile kernel.  Sampled rows against the
    oracle, and the same bits as the kernel forced."""
    h, d = 4, 128
    cases = [([2100, 2500, 3000, 5000, 100, 90, 80], 2),   # mean below 2048: two-tile (table)
             ([300, 17, 256, 129], 2),
             ([40] * 100, 1)]                               # 100 sequences: past the table
    for ls, expect in cases:
        q, k, v, _, cu, _ = sdpa_inputs.packed(ls, ls, h, d, seed=71 + len(ls))
        args = (q.cuda(), k.cuda(), v.cuda(), cu.cuda(), cu.cuda(), max(ls), max(ls))
        sdpa.sdpa_set_forward_variant(0)  # the automatic choice (the module's fixture forces one)
        o, lse = sdpa.attention_varlen(*args, scale=0.088, causal=True)
        sdpa.sdpa_set_forward_variant(expect)
        try:
            o2, lse2 = sdpa.attention_varlen(*args, scale=0.088, causal=True)
        finally:
            sdpa.sdpa_set_forward_variant(0)
        torch.cuda.synchronize()
        assert torch.equal(o, o2) and torch.equal(lse, lse2), f"{len(ls)} sequences"
        o, lse = o.cpu(), lse.cpu()
        cl = cu.tolist()
        for i, L in enumerate(ls[:8]):
            hh = i % h
            a, e = cl[i], cl[i + 1]
            rows = _sampled_rows(L, i + 3)
            ro, rl = oracle.attn_fwd_rows(q[a:e, hh], k[a:e, hh], v[a:e, hh], rows, 0.088, True)
            check_rel(o[a:e, hh][rows], ro, O_TOL[torch.bfloat16], f"o seq {i}")
            check_lse(lse[a:e, hh][rows], rl, f"lse seq {i}")