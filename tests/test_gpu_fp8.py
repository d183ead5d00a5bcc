"""FP8 (E4M3) forward through the C ABI vs the fp64 oracle of the dequantized
inputs (cudnn-frontend PR #554, per-tensor FP8 forward with device descales).

Bounds derived from the arithmetic (the task fixes none for FP8):
- The scores are products of E4M3 values (8 significant bits each, exact in
  fp32) summed in fp32, and the row sums and LSE use the fp32 P, so LSE keeps
  the 16-bit bound |dLSE| <= 1e-3.
- P enters P V rounded to E4M3 (relative error <= 2^-4 per element). O is
  normalised by the fp32 row sum l = sum p_j, so
  |dO_i| <= sum_j 2^-4 p_j |v_j| / l <= 2^-4 max|V|, plus the output rounding
  (bf16: 2^-8 relative; E4M3: 2^-4 relative).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import sdpa_inputs
from helpers import check_lse, np64

pytestmark = pytest.mark.gpu


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


def _scalar(x):
    return torch.tensor([x], dtype=torch.float32, device="cuda")


def _o_bound(vreal_max, oref_max, out_rel):
    return 2.0 ** -4 * vreal_max + out_rel * oref_max + 1e-6


CASES = [
    # b, h, h_kv, s_q, s_kv, mask, window
    (2, 4, 4, 300, 300, "top_left", -1),
    (1, 4, 4, 257, 700, "none", -1),
    (1, 8, 2, 520, 520, "bottom_right", -1),
    (1, 4, 1, 400, 640, "bottom_right", 120),
    (1, 2, 2, 2100, 2100, "top_left", -1),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"b{c[0]}h{c[1]}kv{c[2]}s{c[3]}x{c[4]}_{c[5]}_w{c[6]}")
def test_fp8_dense_bf16_out(sdpa, variant, case):
    b, h, h_kv, s_q, s_kv, mask, window = case
    d = 128
    qc, kc, vc, dq, dk, dv = sdpa_inputs.fp8_dense(b, h, s_q, s_kv, d, seed=9000 + s_q, h_kv=h_kv)
    scale = 1.0 / math.sqrt(d)
    o, lse, amax = sdpa.attention_fp8(qc.cuda(), kc.cuda(), vc.cuda(), _scalar(dq), _scalar(dk),
                                      _scalar(dv), scale=scale, mask=mask, window_left=window)
    torch.cuda.synchronize()
    ro, rlse = oracle.sdpa_fwd_fp8(qc, kc, vc, dq, dk, dv, scale, mask, window)
    vmax = float(np.abs(oracle.e4m3_to_f64(vc, dv)).max())
    err = float(np.abs(np64(o) - ro).max())
    bound = _o_bound(vmax, np.abs(ro).max(), 2.0 ** -8)
    assert err <= bound, f"max|dO| {err:.3e} > bound {bound:.3e}"
    check_lse(lse, rlse)
    # amax: max |O| before the bf16 rounding of the output
    omax = float(o.float().abs().max())
    assert abs(float(amax) - omax) <= 2.0 ** -8 * omax + 1e-12


def test_fp8_e4m3_output_and_amax(sdpa, variant):
    b, h, s, d = 1, 4, 600, 128
    qc, kc, vc, dq, dk, dv = sdpa_inputs.fp8_dense(b, h, s, s, d, seed=91)
    args = (qc.cuda(), kc.cuda(), vc.cuda(), _scalar(dq), _scalar(dk), _scalar(dv))
    scale = 1.0 / math.sqrt(d)
    o16, _, amax16 = sdpa.attention_fp8(*args, scale=scale, causal=True)
    scale_o = 448.0 / float(amax16)  # the next-step scale a caller would pick
    o8, lse8, amax8 = sdpa.attention_fp8(*args, scale=scale, causal=True,
                                         out_dtype=torch.float8_e4m3fn, scale_o=_scalar(scale_o))
    torch.cuda.synchronize()
    assert float(amax8) == float(amax16)  # the same real-valued O, max taken before any rounding
    dec = oracle.e4m3_to_f64(o8, 1.0 / scale_o)
    ref = np64(o16)
    # E4M3 rounding of O * scale_o: relative 2^-4, on top of the bf16 copy's 2^-8
    assert np.all(np.abs(dec - ref) <= 2.0 ** -4 * np.abs(ref) * 1.01 + 2.0 ** -8 * np.abs(ref) + 2.0 ** -9 / scale_o)
    ro, rlse = oracle.sdpa_fwd_fp8(qc, kc, vc, dq, dk, dv, scale, "top_left", -1)
    check_lse(lse8, rlse)


def test_fp8_fp16_output(sdpa, variant):
    b, h, s, d = 1, 2, 333, 128
    qc, kc, vc, dq, dk, dv = sdpa_inputs.fp8_dense(b, h, s, s, d, seed=92)
    scale = 1.0 / math.sqrt(d)
    o, lse, _ = sdpa.attention_fp8(qc.cuda(), kc.cuda(), vc.cuda(), _scalar(dq), _scalar(dk),
                                   _scalar(dv), scale=scale, causal=True, out_dtype=torch.float16)
    torch.cuda.synchronize()
    assert o.dtype == torch.float16
    ro, rlse = oracle.sdpa_fwd_fp8(qc, kc, vc, dq, dk, dv, scale, "top_left", -1)
    vmax = float(np.abs(oracle.e4m3_to_f64(vc, dv)).max())
    assert float(np.abs(np64(o) - ro).max()) <= _o_bound(vmax, np.abs(ro).max(), 2.0 ** -11)
    check_lse(lse, rlse)


def test_fp8_packed(sdpa, variant):
    lq = [130, 7, 300, 64, 0]
    lk = [130, 40, 300, 64, 9]
    h, h_kv, d = 4, 2, 128
    qc, kc, vc, dq, dk, dv, cu_q, cu_kv = sdpa_inputs.fp8_packed(lq, lk, h, d, seed=93, h_kv=h_kv)
    scale = 1.0 / math.sqrt(d)
    T = qc.shape[0]
    o = torch.empty(T, h, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(T, h, dtype=torch.float32, device="cuda")
    amax = torch.empty(1, dtype=torch.float32, device="cuda")
    sdpa.sdpa_varlen_fwd_fp8(qc.cuda(), kc.cuda(), vc.cuda(), o, lse, _scalar(dq), _scalar(dk),
                             _scalar(dv), None, amax, cu_q.cuda(), cu_kv.cuda(), len(lq), T,
                             kc.shape[0], max(lq), max(lk), h, h_kv, d, scale, 2, -1, 0)
    torch.cuda.synchronize()
    ro, rlse = oracle.sdpa_varlen_fwd_fp8(qc, kc, vc, cu_q, cu_kv, dq, dk, dv, scale, "bottom_right")
    vmax = float(np.abs(oracle.e4m3_to_f64(vc, dv)).max())
    assert float(np.abs(np64(o) - ro).max()) <= _o_bound(vmax, np.abs(ro).max(), 2.0 ** -8)
    check_lse(lse, rlse)


def test_fp8_rms_error_within_the_statistical_bound(sdpa, variant):
    # Round-to-nearest errors of P are independent with RMS <= 2^-4 / sqrt(3)
    # (uniform within half an E4M3 step), so E[dO_i^2] <= (2^-4/sqrt(3))^2 *
    # sum_j (p_j/l)^2 v_j^2 <= (2^-4/sqrt(3))^2 * max_j v_j^2-weighted mean:
    # over all rows, RMS(dO) <= 2^-4/sqrt(3) * RMS(V) for these inputs.
    b, h, s, d = 1, 4, 1024, 128
    qc, kc, vc, dq, dk, dv = sdpa_inputs.fp8_dense(b, h, s, s, d, seed=94)
    scale = 1.0 / math.sqrt(d)
    o, _, _ = sdpa.attention_fp8(qc.cuda(), kc.cuda(), vc.cuda(), _scalar(dq), _scalar(dk),
                                 _scalar(dv), scale=scale, causal=True)
    torch.cuda.synchronize()
    ro, _ = oracle.sdpa_fwd_fp8(qc, kc, vc, dq, dk, dv, scale, "top_left", -1)
    rms = float(np.sqrt(np.mean((np64(o) - ro) ** 2)))
    vrms = float(np.sqrt(np.mean(oracle.e4m3_to_f64(vc, dv) ** 2)))
    assert rms <= 2.0 ** -4 / math.sqrt(3) * vrms, (rms, vrms)


def test_fp8_validation(sdpa):
    from scaled_dot_product_04_gb300 import _lib as L
    q = torch.empty(1, 1, 128, 64, dtype=torch.uint8, device="cuda")
    o = torch.empty(1, 1, 128, 64, dtype=torch.bfloat16, device="cuda")
    one = _scalar(1.0)
    with pytest.raises(sdpa.SdpaError) as e:
        sdpa.sdpa_fwd_fp8(q, q, q, o, None, one, one, one, None, None, 1, 1, 1, 128, 128, 64, 0.1,
                          1, -1, 0)
    assert e.value.status == L.SDPA_ERR_UNSUPPORTED and "d = 128" in str(e.value)
    q = torch.empty(1, 1, 128, 128, dtype=torch.uint8, device="cuda")
    with pytest.raises(sdpa.SdpaError) as e:  # E4M3 output without scale_o
        sdpa.sdpa_fwd_fp8(q, q, q, o, None, one, one, one, None, None, 1, 1, 1, 128, 128, 128, 0.1,
                          1, -1, 2)
    assert e.value.status == L.SDPA_ERR_INVALID_ARG and "scale_o" in str(e.value)
    with pytest.raises(sdpa.SdpaError) as e:
        sdpa.sdpa_fwd_fp8(q, q, q, o, None, None, one, one, None, None, 1, 1, 1, 128, 128, 128, 0.1,
                          1, -1, 0)
    assert e.value.status == L.SDPA_ERR_INVALID_ARG
