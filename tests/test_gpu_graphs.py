"""The forward and backward chains captured in a CUDA graph (torch.cuda.graph)
and replayed on new inputs copied into the captured buffers: every launch of
the library is a plain stream operation -- the programmatically overlapped
launches of the backward chain, the counter reset of the dynamically
scheduled forwards, the persistent backward's counter zeroed by its
preprocess kernel -- so a replay gives the eager calls' results: O, LSE, dK
and dV bit for bit, dQ to rounding (its fp32 additions may arrive in another
order)."""
import math

import pytest
import torch

import sdpa_inputs
from helpers import check_rel

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sdpa():
    import scaled_dot_product_04_gb300 as m
    m.load()
    return m


def _same(a, b, name):
    assert torch.equal(a, b), f"{name} differs from the eager call"


def _replays(capture, inputs, draws, eager):
    """Capture `capture()` once on the static `inputs`, then for each draw copy
    it into them, replay, and compare with `eager(draw)`."""
    for _ in range(2):  # warm-up: first-call set-up happens outside the capture
        capture()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        outs = capture()
    for draw in draws:
        for dst, src in zip(inputs, draw):
            dst.copy_(src)
        g.replay()
        torch.cuda.synchronize()
        ref = eager(draw)
        torch.cuda.synchronize()
        yield outs, ref


@pytest.mark.parametrize("b,h,s,d,causal", [
    (4, 16, 1024, 64, True),     # backward on the persistent kernel
    (2, 8, 4096, 128, False),    # two-tile forward with a cut tail when the SM count leaves one; one CTA per key tile
])
def test_dense_chain_in_a_graph(sdpa, b, h, s, d, causal):
    scale = 1.0 / math.sqrt(d)
    draws = [tuple(x.cuda() for x in sdpa_inputs.dense(b, h, s, s, d, seed=seed)) for seed in (1, 2)]
    q, k, v, do = (torch.empty_like(x) for x in draws[0])

    def chain(q, k, v, do):
        o, lse = sdpa.attention(q, k, v, scale=scale, causal=causal)
        dq, dk, dv = sdpa.attention_bwd(q, k, v, o, do, lse, scale=scale, causal=causal)
        return o, lse, dq, dk, dv

    for outs, ref in _replays(lambda: chain(q, k, v, do), (q, k, v, do), draws, lambda dr: chain(*dr)):
        for name, a, r in zip(("o", "lse", "dq", "dk", "dv"), outs, ref):
            if name == "dq":
                check_rel(a, r.double().cpu().numpy(), 1e-2, "dq vs eager")
            else:
                _same(a, r, name)


def test_packed_chain_in_a_graph(sdpa):
    lens = [700, 1300, 90, 2500, 400, 1, 1900, 640]
    h, d = 8, 128
    draws = []
    for seed in (3, 4):
        q, k, v, do, cu, _ = sdpa_inputs.packed(lens, lens, h, d, seed=seed)
        draws.append((q.cuda(), k.cuda(), v.cuda(), do.cuda()))
    cu = cu.cuda()
    q, k, v, do = (torch.empty_like(x) for x in draws[0])
    m = max(lens)

    def chain(q, k, v, do):
        o, lse = sdpa.attention_varlen(q, k, v, cu, cu, m, m, scale=0.088, causal=True)
        dq, dk, dv = sdpa.attention_varlen_bwd(q, k, v, o, do, lse, cu, cu, m, m, scale=0.088, causal=True)
        return o, lse, dq, dk, dv

    for outs, ref in _replays(lambda: chain(q, k, v, do), (q, k, v, do), draws, lambda dr: chain(*dr)):
        for name, a, r in zip(("o", "lse", "dq", "dk", "dv"), outs, ref):
            if name == "dq":
                check_rel(a, r.double().cpu().numpy(), 1e-2, "dq vs eager")
            else:
                _same(a, r, name)
