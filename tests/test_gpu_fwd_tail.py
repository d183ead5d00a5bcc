"""The two-tile forward's tail split: a dense list of equal units (no mask, no
window) whose count leaves a partial last wave on the grid runs its last units
as 128-row halves.  Here the head count is chosen from the device's SM count
so that the last wave is partial and at most half full, which makes the host
cut it; rows of a cut unit's second half, of the next unit's rows and of a
ragged last block must all come out right.

Tolerances: O within 1e-2 of max|O_ref| (16-bit), LSE within 1e-3; FP8 within
the derived bound of tests/test_gpu_fp8.py (2^-4 max|V| + 2^-8 max|O_ref|).
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
    m.sdpa_set_forward_variant(2)
    yield m
    m.sdpa_set_forward_variant(0)


def _heads(s):
    """A head count whose 256-row units (b = 1) overrun the SMs by at most half a wave."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    blocks = (s + 255) // 256
    h = sms // blocks + 1
    units = blocks * h
    rest = units % sms
    assert units > sms and 0 < 2 * rest <= sms, (sms, blocks, h)
    return h


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("s", [1024, 1000, 770, 600])
def test_split_tail_dense(sdpa, d, s):
    h = _heads(s)
    q, k, v, _ = sdpa_inputs.dense(1, h, s, s, d, seed=300 + s + d)
    scale = 1.0 / math.sqrt(d)
    o, lse = sdpa.attention(q.cuda(), k.cuda(), v.cuda(), scale=scale, causal=False)
    torch.cuda.synchronize()
    ro, rlse = oracle.sdpa_fwd(q, k, v, scale, False)
    check_rel(o, ro, O_TOL[torch.bfloat16], "o")
    check_lse(lse, rlse)
    for hh in (0, h - 1):  # whole heads on both ends of the list
        check_rel(o[0, hh], ro[0, hh], O_TOL[torch.bfloat16], f"o head {hh}")


def test_split_tail_fp16_gqa(sdpa):
    s, d = 1000, 128
    h = _heads(s)
    h += h % 2  # two query heads per key/value head
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    units = 4 * h
    if not (units > sms and 0 < 2 * (units % sms) <= sms):
        pytest.skip("no partial last wave at this SM count")
    q, k, v, _ = sdpa_inputs.dense(1, h, s, s, d, seed=77, dtype=torch.float16, h_kv=h // 2)
    scale = 1.0 / math.sqrt(d)
    o, lse = sdpa.attention(q.cuda(), k.cuda(), v.cuda(), scale=scale, mask="none")
    torch.cuda.synchronize()
    ro, rlse = oracle.sdpa_fwd_ex(q, k, v, scale, "none", -1)
    check_rel(o, ro, O_TOL[torch.float16], "o")
    check_lse(lse, rlse)


def _sc(x):
    return torch.tensor([x], dtype=torch.float32, device="cuda")


def test_split_tail_fp8(sdpa):
    s, d = 1000, 128
    h = _heads(s)
    qc, kc, vc, dq, dk, dv = sdpa_inputs.fp8_dense(1, h, s, s, d, seed=9100)
    o, lse, _ = sdpa.attention_fp8(qc.cuda(), kc.cuda(), vc.cuda(), _sc(dq), _sc(dk), _sc(dv),
                                   scale=1.0 / math.sqrt(d), mask="none")
    torch.cuda.synchronize()
    ro, rlse = oracle.sdpa_fwd_fp8(qc, kc, vc, dq, dk, dv, 1.0 / math.sqrt(d), "none", -1)
    vmax = float(np.abs(oracle.e4m3_to_f64(vc, dv)).max())
    err = float(np.abs(np64(o) - ro).max())
    bound = 2.0 ** -4 * vmax + 2.0 ** -8 * float(np.abs(ro).max()) + 1e-6
    assert err <= bound, f"max|dO| {err:.3e} > bound {bound:.3e}"
    check_lse(lse, rlse)


def test_split_tail_fp8_fp16_and_e4m3_outputs(sdpa):
    """The other output kinds of the cut-tail FP8 instantiations: fp16 against
    the oracle, E4M3 (O x scale_o) against the bf16 output of the same call."""
    s, d = 770, 128
    h = _heads(s)
    qc, kc, vc, dq, dk, dv = sdpa_inputs.fp8_dense(1, h, s, s, d, seed=9101)
    args = (qc.cuda(), kc.cuda(), vc.cuda(), _sc(dq), _sc(dk), _sc(dv))
    scale = 1.0 / math.sqrt(d)
    o16, _, amax16 = sdpa.attention_fp8(*args, scale=scale, mask="none")
    oh, lseh, _ = sdpa.attention_fp8(*args, scale=scale, mask="none", out_dtype=torch.float16)
    scale_o = 448.0 / float(amax16)
    o8, lse8, amax8 = sdpa.attention_fp8(*args, scale=scale, mask="none",
                                         out_dtype=torch.float8_e4m3fn, scale_o=_sc(scale_o))
    torch.cuda.synchronize()
    ro, rlse = oracle.sdpa_fwd_fp8(qc, kc, vc, dq, dk, dv, scale, "none", -1)
    vmax = float(np.abs(oracle.e4m3_to_f64(vc, dv)).max())
    bound = 2.0 ** -4 * vmax + 2.0 ** -11 * float(np.abs(ro).max()) + 1e-6
    assert float(np.abs(np64(oh) - ro).max()) <= bound
    check_lse(lseh, rlse)
    assert float(amax8) == float(amax16)
    dec = oracle.e4m3_to_f64(o8, 1.0 / scale_o)
    ref = np64(o16)
    assert np.all(np.abs(dec - ref) <= 2.0 ** -4 * np.abs(ref) * 1.01 + 2.0 ** -8 * np.abs(ref) + 2.0 ** -9 / scale_o)
    check_lse(lse8, rlse)
