"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no attention arithmetic: it only draws tensors.  Both the
CUDA path and the fp64 oracle consume exactly the tensors drawn here, so the
two sides see bit-identical inputs.

Recipe (the pages fix none of it beyond the shapes):
  * fp32 ``torch.randn`` from ``torch.Generator().manual_seed(seed)`` on the
    CPU, drawn in the order Q, K, V, dO, then rounded to the I/O dtype (RNE);
  * the long-context workload multiplies the rounded Q and K by 2, which is
    exact in bf16/fp16;
  * varlen lengths are integers uniform on [64, 4096] drawn with
    ``torch.randint`` from seed 2004; q and kv share the lengths.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    layout: str            # "bhsd" or "thd"
    b: int = 1             # batch (dense) / number of sequences (thd)
    h: int = 1
    s: int = 0             # dense sequence length (s_q == s_kv)
    d: int = 64
    causal: bool = True
    qk_mult: float = 1.0
    backward: bool = False
    seed: int = 0
    len_seed: int = 0      # thd only
    len_lo: int = 64
    len_hi: int = 4096
    extra: dict = field(default_factory=dict, compare=False)

    @property
    def scale(self) -> float:
        return 1.0 / float(self.d) ** 0.5


# The five workloads the pages' shapes and the task configuration define.
WORKLOADS = {
    "c1_b1h2s128d64_causal": Workload("c1_b1h2s128d64_causal", "bhsd", b=1, h=2, s=128, d=64,
                                      causal=True, seed=1001),
    "c2_b4h16s1024d64_causal": Workload("c2_b4h16s1024d64_causal", "bhsd", b=4, h=16, s=1024,
                                        d=64, causal=True, seed=1002),
    "c3_b2h16s4096d128_noncausal": Workload("c3_b2h16s4096d128_noncausal", "bhsd", b=2, h=16,
                                            s=4096, d=128, causal=False, backward=True,
                                            seed=1003),
    "c4_thd16_h32d128_causal": Workload("c4_thd16_h32d128_causal", "thd", b=16, h=32, d=128,
                                        causal=True, backward=True, seed=1004, len_seed=2004),
    "c5_b1h32s16384d128_causal_qk2": Workload("c5_b1h32s16384d128_causal_qk2", "bhsd", b=1,
                                              h=32, s=16384, d=128, causal=True, qk_mult=2.0,
                                              backward=True, seed=1005),
}


def _draw(shapes, seed: int, dtype: torch.dtype):
    g = torch.Generator().manual_seed(seed)
    return [torch.randn(shape, generator=g, dtype=torch.float32).to(dtype) for shape in shapes]


def dense(b: int, h: int, s_q: int, s_kv: int, d: int, seed: int,
          dtype: torch.dtype = torch.bfloat16, qk_mult: float = 1.0, h_kv: int | None = None):
    """Q [b,h,s_q,d], K/V [b,h_kv,s_kv,d] (h_kv defaults to h), dO [b,h,s_q,d] on the CPU."""
    hk = h if h_kv is None else h_kv
    q, k, v, do = _draw([(b, h, s_q, d), (b, hk, s_kv, d), (b, hk, s_kv, d), (b, h, s_q, d)],
                        seed, dtype)
    if qk_mult != 1.0:
        q = q * qk_mult
        k = k * qk_mult
    return q, k, v, do


def varlen_lengths(n: int, seed: int, lo: int = 64, hi: int = 4096) -> list[int]:
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, (n,), generator=g).tolist()


def cu_seqlens(lengths) -> torch.Tensor:
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + int(L))
    return torch.tensor(cu, dtype=torch.int32)


def packed(lengths_q, lengths_kv, h: int, d: int, seed: int,
           dtype: torch.dtype = torch.bfloat16, qk_mult: float = 1.0, h_kv: int | None = None):
    """THD tensors: Q/dO [Tq,h,d], K/V [Tkv,h_kv,d] (h_kv defaults to h) and the two cu_seqlens."""
    hk = h if h_kv is None else h_kv
    tq, tkv = int(sum(lengths_q)), int(sum(lengths_kv))
    q, k, v, do = _draw([(tq, h, d), (tkv, hk, d), (tkv, hk, d), (tq, h, d)], seed, dtype)
    if qk_mult != 1.0:
        q = q * qk_mult
        k = k * qk_mult
    return q, k, v, do, cu_seqlens(lengths_q), cu_seqlens(lengths_kv)


def make(w: Workload, dtype: torch.dtype = torch.bfloat16):
    """All inputs of a named workload as a dict of CPU tensors."""
    if w.layout == "bhsd":
        q, k, v, do = dense(w.b, w.h, w.s, w.s, w.d, w.seed, dtype, w.qk_mult)
        return dict(q=q, k=k, v=v, do=do)
    lens = varlen_lengths(w.b, w.len_seed, w.len_lo, w.len_hi)
    q, k, v, do, cu_q, cu_kv = packed(lens, lens, w.h, w.d, w.seed, dtype, w.qk_mult)
    return dict(q=q, k=k, v=v, do=do, cu_q=cu_q, cu_kv=cu_kv, lengths=lens)



def fp8_quantize(x: torch.Tensor):
    """Per-tensor E4M3 encoding of a synthetic tensor: codes (uint8) of x * s
    with s = 448 / max|x| (the largest code maps to the largest magnitude),
    and the descale 1 / s as a float.  Input generation only."""
    amax = float(x.abs().max())
    s = 448.0 / amax if amax > 0 else 1.0
    codes = (x.float() * s).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, 1.0 / s


def fp8_dense(b: int, h: int, s_q: int, s_kv: int, d: int, seed: int, h_kv: int | None = None):
    """E4M3 codes of Q [b,h,s_q,d], K/V [b,h_kv,s_kv,d] drawn N(0,1), with their descales."""
    q, k, v, _ = dense(b, h, s_q, s_kv, d, seed, torch.float32, h_kv=h_kv)
    (qc, dq), (kc, dk), (vc, dv) = fp8_quantize(q), fp8_quantize(k), fp8_quantize(v)
    return qc, kc, vc, dq, dk, dv


def fp8_packed(lengths_q, lengths_kv, h: int, d: int, seed: int, h_kv: int | None = None):
    """E4M3 codes of packed Q/K/V, their descales and the two cu_seqlens."""
    q, k, v, _, cu_q, cu_kv = packed(lengths_q, lengths_kv, h, d, seed, torch.float32, h_kv=h_kv)
    (qc, dq), (kc, dk), (vc, dv) = fp8_quantize(q), fp8_quantize(k), fp8_quantize(v)
    return qc, kc, vc, dq, dk, dv, cu_q, cu_kv
