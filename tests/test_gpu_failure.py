"""Failure detection on the GPU without a GPU fault, and guarded outputs.

- A bounded wait that expires: the self-test kernel polls, with the same
  bounded wait every kernel uses (here limited to 20 ms), a barrier phase that
  nothing completes.  The wait gives up, records its kernel and site in the
  error word and the kernel exits; sdpa_check_device_error reports
  SDPA_ERR_TIMEOUT, clears the word, and the context stays usable.
- Canary regions around every output of the backward, the extended calls and
  the FP8 forward stay untouched (a write past an output's end would show).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import sdpa_inputs
from helpers import GRAD_TOL, O_TOL, check_rel

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sdpa():
    import scaled_dot_product_04_gb300 as m
    m.load()
    return m


def test_an_expired_wait_reports_timeout_and_the_context_survives(sdpa):
    from scaled_dot_product_04_gb300 import _lib as L
    sdpa.sdpa_check_device_error()  # nothing pending
    sdpa.sdpa_selftest_wait_timeout(20000)
    with pytest.raises(sdpa.SdpaError) as e:
        sdpa.sdpa_check_device_error()
    assert e.value.status == L.SDPA_ERR_TIMEOUT
    assert "selftest" in str(e.value) and "site 1" in str(e.value)
    sdpa.sdpa_check_device_error()  # the word was cleared
    # the context still computes correct results
    q, k, v, _ = sdpa_inputs.dense(1, 2, 200, 200, 64, seed=3)
    o, lse = sdpa.attention(q.cuda(), k.cuda(), v.cuda(), scale=0.125, causal=True)
    torch.cuda.synchronize()
    ro, _ = oracle.sdpa_fwd(q, k, v, 0.125, True)
    check_rel(o, ro, O_TOL[torch.bfloat16], "o after the self-test")
    sdpa.sdpa_check_device_error()


def test_selftest_rejects_a_bad_limit(sdpa):
    with pytest.raises(sdpa.SdpaError):
        sdpa.sdpa_selftest_wait_timeout(0)


def _guarded(shape, dtype, fill, guard=4096):
    n = int(np.prod(shape))
    buf = torch.full((n + 2 * guard,), fill, dtype=dtype, device="cuda")
    return buf, buf[guard:guard + n].view(*shape), guard


def _untouched(buf, guard, fill):
    head, tail = buf[:guard], buf[-guard:]
    if isinstance(fill, float) and math.isnan(fill):
        return bool(torch.isnan(head.float()).all() and torch.isnan(tail.float()).all())
    return bool((head == fill).all() and (tail == fill).all())


@pytest.mark.parametrize("deterministic", [0, 1])
def test_backward_outputs_and_workspace_are_guarded(sdpa, deterministic):
    b, h, h_kv, s, d = 1, 4, 2, 333, 128
    q, k, v, do = (x.cuda() for x in sdpa_inputs.dense(b, h, s, s, d, seed=71, h_kv=h_kv))
    scale = 1.0 / math.sqrt(d)
    o, lse = sdpa.attention(q, k, v, scale=scale, causal=True)
    nan = float("nan")
    bufs = [_guarded(x.shape, x.dtype, nan) for x in (q, k, v)]
    need = sdpa.sdpa_bwd_ex_workspace_size(b, h, s, d, deterministic)
    wsb, ws, wg = _guarded((need,), torch.uint8, 0xA5)
    sdpa.sdpa_bwd_ex(q, k, v, o, do, lse, bufs[0][1], bufs[1][1], bufs[2][1], b, h, h_kv, s, s, d,
                     scale, 1, -1, deterministic, 0, ws, need)
    torch.cuda.synchronize()
    for name, (buf, _, g) in zip(("dq", "dk", "dv"), bufs):
        assert _untouched(buf, g, nan), name
    assert _untouched(wsb, wg, 0xA5), "workspace"
    ref = oracle.sdpa_bwd_ex(q, k, v, do, scale, "top_left", -1)
    for name, (_, x, _), r in zip(("dq", "dk", "dv"), bufs, ref):
        check_rel(x, r, GRAD_TOL, name)


def test_fp8_outputs_are_guarded(sdpa):
    b, h, s, d = 1, 2, 300, 128
    qc, kc, vc, dq, dk, dv = sdpa_inputs.fp8_dense(b, h, s, s, d, seed=72)
    sc = [torch.tensor([x], dtype=torch.float32, device="cuda") for x in (dq, dk, dv, 8.0)]
    ob, o, og = _guarded((b, h, s, d), torch.uint8, 0x7F)           # E4M3 output, NaN code fill
    lb, lse, lg = _guarded((b, h, s), torch.float32, 12345.0)
    ab, amax, ag = _guarded((1,), torch.float32, -7.0, guard=16)
    sdpa.sdpa_fwd_fp8(qc.cuda(), kc.cuda(), vc.cuda(), o, lse, sc[0], sc[1], sc[2], sc[3], amax, b,
                      h, h, s, s, d, 1.0 / math.sqrt(d), 1, -1, 2)
    torch.cuda.synchronize()
    assert _untouched(ob, og, 0x7F) and _untouched(lb, lg, 12345.0) and _untouched(ab, ag, -7.0)
    assert float(amax) > 0
