"""Full-size parity of the other timed configurations of the long workload.

The long causal workload (b1 h32 s16384 d128, Q and K doubled) run exactly as
the benchmark's variants launch it:
- the backward with its deterministic dQ pass: whole heads 0, 3, 4 and 31 of
  dQ/dK/dV against the fp64 oracle (tolerance 2e-2 of max|ref| per tensor),
  and a bit-identical rerun;
- the FP8 (E4M3) forward with per-tensor descales and bf16 output: whole heads
  0, 16 and 31 of O within the derived bound 2^-4 max|V| + 2^-8 max|O_ref| of
  the oracle on the decoded inputs, LSE within 1e-3;
- the extended-call rows: whole heads under the left window and the
  bottom-right mask, sampled rows of one key/value head group for GQA.
"""
import numpy as np
import pytest
import torch

import oracle
import oracle_refs
import sdpa_inputs
from helpers import GRAD_TOL, check_lse, check_rel, np64

pytestmark = pytest.mark.gpu

NAME = "c5_b1h32s16384d128_causal_qk2"


@pytest.fixture(scope="module")
def sdpa():
    import scaled_dot_product_04_gb300 as m
    m.load()
    return m


def _rows(n, seed):
    g = np.random.default_rng(seed)
    base = {0, 1, 127, 128, n // 2, n - 129, n - 128, n - 1}
    base |= set(g.integers(0, n, 6).tolist())
    return np.array(sorted(r for r in base if 0 <= r < n), np.int32)


@pytest.mark.usefixtures("bwd_kernel")
def test_full_size_deterministic_bwd_whole_heads_and_bitwise(sdpa):
    w = sdpa_inputs.WORKLOADS[NAME]
    t = oracle_refs.inputs(NAME)
    q, k, v, do = (t[x].cuda() for x in ("q", "k", "v", "do"))
    o, lse = sdpa.attention(q, k, v, scale=w.scale, causal=True)
    ws = torch.empty(sdpa.sdpa_bwd_ex_workspace_size(w.b, w.h, w.s, w.d, 1), dtype=torch.uint8,
                     device="cuda")
    g1 = sdpa.attention_bwd(q, k, v, o, do, lse, scale=w.scale, causal=True, deterministic=True,
                            workspace=ws)
    g2 = sdpa.attention_bwd(q, k, v, o, do, lse, scale=w.scale, causal=True, deterministic=True,
                            workspace=ws)
    torch.cuda.synchronize()
    for a, b, name in zip(g1, g2, ("dq", "dk", "dv")):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), f"{name} differs on rerun"
    dq, dk, dv = (x.cpu() for x in g1)
    del g1, g2
    for hh in (0, 3, 4, w.h - 1):
        r = oracle_refs.dense_slice(NAME, 0, hh, True)
        for g, rr, nm in zip((dq, dk, dv), r[2:], ("dq", "dk", "dv")):
            check_rel(g[0, hh], rr, GRAD_TOL, f"{nm}[{hh}]")


def test_full_size_fp8_fwd_whole_heads(sdpa):
    w = sdpa_inputs.WORKLOADS[NAME]
    t = oracle_refs.inputs(NAME)
    enc = [sdpa_inputs.fp8_quantize(t[x].float()) for x in ("q", "k", "v")]
    (qc, dsq), (kc, dsk), (vc, dsv) = enc
    ds = [torch.tensor([x], dtype=torch.float32, device="cuda") for x in (dsq, dsk, dsv)]
    o, lse, amax = sdpa.attention_fp8(qc.cuda(), kc.cuda(), vc.cuda(), *ds, scale=w.scale,
                                      causal=True)
    torch.cuda.synchronize()
    o, lse = o.cpu(), lse.cpu()
    assert torch.isfinite(o.float()).all()
    for hh in (0, w.h // 2, w.h - 1):
        qd = oracle.e4m3_to_f64(qc[0:1, hh:hh + 1], dsq)
        kd = oracle.e4m3_to_f64(kc[0:1, hh:hh + 1], dsk)
        vd = oracle.e4m3_to_f64(vc[0:1, hh:hh + 1], dsv)
        ro, rlse = oracle.sdpa_fwd(qd, kd, vd, w.scale, True)
        err = float(np.abs(np64(o[0, hh]) - ro[0, 0]).max())
        bound = 2.0 ** -4 * float(np.abs(vd).max()) + 2.0 ** -8 * float(np.abs(ro).max()) + 1e-6
        assert err <= bound, f"head {hh}: max|dO| {err:.3e} > bound {bound:.3e}"
        check_lse(lse[0, hh], rlse[0, 0], f"lse[{hh}]")


# The extended-call rows as bench.py runs them on the long workload: 8
# key/value heads; causal with window_left = 2048; 4096 queries against the
# 16384 keys under the bottom-right mask.  O, LSE, dQ, dK, dV against the
# oracle's extended definitions: a whole head for the window and the
# bottom-right mask; sampled rows of one key/value head's group for GQA (a
# key/value head's dK and dV sum over its group's query heads).
EXT = {"gqa": (8, 16384, "top_left", -1),
       "window": (32, 16384, "top_left", 2048),
       "bottom_right": (32, 4096, "bottom_right", -1)}


@pytest.mark.parametrize("name", list(EXT))
def test_full_size_extended_rows(sdpa, name):
    from helpers import O_TOL
    w = sdpa_inputs.WORKLOADS[NAME]
    h_kv, s_q, mask, window = EXT[name]
    q, k, v, do = sdpa_inputs.dense(w.b, w.h, s_q, w.s, w.d, w.seed, qk_mult=w.qk_mult,
                                    h_kv=h_kv)
    qg, kg, vg, dog = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = sdpa.attention(qg, kg, vg, scale=w.scale, mask=mask, window_left=window)
    dq, dk, dv = sdpa.attention_bwd(qg, kg, vg, o, dog, lse, scale=w.scale, mask=mask,
                                    window_left=window)
    torch.cuda.synchronize()
    o, lse, dq, dk, dv = (x.cpu() for x in (o, lse, dq, dk, dv))
    del qg, kg, vg, dog
    group = w.h // h_kv
    hk = min(1, h_kv - 1)
    heads = [hk * group + g for g in range(group)]
    if group == 1:
        # one query head per key/value head: the whole head, every row
        hh = heads[0]
        sl = [x[0:1, hh:hh + 1] for x in (q, k, v, do)]
        ro, rl = oracle.sdpa_fwd_ex(sl[0], sl[1], sl[2], w.scale, mask, window)
        check_rel(o[0, hh], ro[0, 0], O_TOL[torch.bfloat16], f"o[{hh}]")
        check_lse(lse[0, hh], rl[0, 0], f"lse[{hh}]")
        r = oracle.sdpa_bwd_ex(*sl, w.scale, mask, window)
        for g, rr, nm in zip((dq, dk, dv), r, ("dq", "dk", "dv")):
            check_rel(g[0, hh], rr[0, 0], GRAD_TOL, f"{nm}[{hh}]")
        return
    qr, kr = _rows(s_q, 7), _rows(w.s, 8)
    r_dk = r_dv = 0
    for hh in heads:
        ro, rl = oracle.attn_fwd_rows_ex(q[0, hh], k[0, hk], v[0, hk], qr, w.scale, mask, window)
        check_rel(o[0, hh][qr], ro, O_TOL[torch.bfloat16], f"o[{hh}]")
        check_lse(lse[0, hh][qr], rl, f"lse[{hh}]")
        g_dq, g_dk, g_dv = oracle.attn_bwd_rows_ex(q[0, hh], k[0, hk], v[0, hk], do[0, hh], qr,
                                                   kr, w.scale, mask, window)
        check_rel(dq[0, hh][qr], g_dq, GRAD_TOL, f"dq[{hh}]")
        r_dk, r_dv = r_dk + g_dk, r_dv + g_dv
    check_rel(dk[0, hk][kr], r_dk, GRAD_TOL, f"dk[{hk}]")
    check_rel(dv[0, hk][kr], r_dv, GRAD_TOL, f"dv[{hk}]")
