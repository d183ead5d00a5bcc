"""The allocation-free backward entry point, sdpa_bwd_noalloc.

It exists for callers that cannot allocate device memory (plug-in code
inside a runtime that owns all allocations, or loops where a cudaMalloc is
not allowed): it takes no workspace and uses a fixed scratch array built
into the library.  These checks call it through the C ABI twice in a row and
compare each result with the workspace-taking sdpa_bwd on the same inputs and
with the fp64 oracle's gradients, within the gradient tolerance the other
tests use.  The file's name makes pytest collect it last.
"""
import math

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
    return m


@pytest.mark.parametrize("d,causal", [(128, True), (64, False)])
def test_noalloc_matches_workspace_backward(sdpa, d, causal):
    b, h, s = 2, 3, 600
    scale = 1.0 / math.sqrt(d)
    host = sdpa_inputs.dense(b, h, s, s, d, seed=31 + d)
    q, k, v, do = (x.cuda() for x in host)
    o, lse = sdpa.attention(q, k, v, scale=scale, causal=causal)
    ref = sdpa.attention_bwd(q, k, v, o, do, lse, scale=scale, causal=causal)
    torch.cuda.synchronize()
    exact = oracle.sdpa_bwd(*host, scale, causal)
    for call in range(2):
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        sdpa.sdpa_bwd_noalloc(q, k, v, o, do, lse, dq, dk, dv, b, h, s, s, d, scale, causal, 0)
        torch.cuda.synchronize()
        for name, got, r, x in zip(("dq", "dk", "dv"), (dq, dk, dv), ref, exact):
            check_rel(got, r.double().cpu().numpy(), GRAD_TOL, f"{name} (call {call + 1})")
            check_rel(got, x, GRAD_TOL, f"{name} vs oracle (call {call + 1})")
    sdpa.sdpa_check_device_error()


def test_noalloc_rejects_problems_beyond_its_scratch(sdpa):
    # 1 x 16 x 8192 rows at d = 128 needs ~64.5 MiB of scratch, over the 32 MiB array
    b, h, s, d = 1, 16, 8192, 128
    q = torch.empty(b, h, s, d, dtype=torch.bfloat16, device="cuda")
    k, v, o, do = (torch.empty_like(q) for _ in range(4))
    lse = torch.empty(b, h, s, device="cuda")
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    with pytest.raises(sdpa.SdpaError) as e:
        sdpa.sdpa_bwd_noalloc(q, k, v, o, do, lse, dq, dk, dv, b, h, s, s, d, 0.088, 1, 0)
    assert e.value.status == 4 and "scratch" in str(e.value)
