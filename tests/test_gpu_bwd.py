"""Backward parity: dq, dk, dv from csattn_attn_bwd against the float64 oracle's
gradients (oracle.attn.attention_backward) on the same bf16 inputs.

Tolerance (bf16).  The parity bounds, max-abs 2e-2 and relative L2 5e-3,
with one allowance: the gradients are returned in bf16, and where their entries
exceed the attention output's range (|dv| reaches ~10 on these inputs) the
rounding of the stored value alone is up to half a bf16 ulp, 2^(e-8) for an entry
in [2^e, 2^(e+1)): 0.031 at 8..16, more than 2e-2 by itself.  So the max-abs bound
is 2e-2 plus half an ulp of the largest reference entry; below 4 that adds at
most 2^-7.  The kernels also round P and dS to bf16 for the tensor-core products
(relative 2^-9 each, independent across terms), which puts the relative L2 error
at ~2.5e-3.  The relative L2 is taken against max(||ref||, 1e-3 sqrt(n)): where the
exact gradient is zero (T = 1, a single key: dP and D = rowsum(dO o O) are the same
dot product summed in different orders, so dS = P (dP - D) is fp32 rounding noise)
it bounds the RMS error by 5e-6 instead of dividing by zero."""
import math

import numpy as np
import pytest
import torch

import attn_workloads as W
import transformer_causal_self_gb300 as csattn
from oracle import attn as OA
from tests.gpu_helpers import assert_grad_close as _close
from tests.gpu_helpers import dev, to_np

pytestmark = pytest.mark.gpu


def _run(q, k, v, do, causal, base, layout, scale):
    qd, kd, vd, dod = (t.to(dev()) for t in (q, k, v, do))
    B, Hq, T, d = q.shape
    lse = torch.empty(B, Hq, T, dtype=torch.float32, device=dev())
    out = csattn.attn_fwd(qd, kd, vd, causal=causal, rope_base=base, rope_layout=layout,
                          scale=scale, lse=lse)
    dq, dk, dv = csattn.attn_bwd(qd, kd, vd, out, dod, lse, causal=causal, rope_base=base,
                                 rope_layout=layout, scale=scale)
    csattn.check_status()
    return dq, dk, dv


CASES = [
    # (B, Hq, Hkv, T, d, causal, rope_base, layout)
    (2, 4, 2, 200, 128, True, 10000.0, "split_half"),
    (1, 3, 3, 130, 64, False, 10000.0, "adjacent"),
    (2, 8, 1, 64, 128, True, 0.0, "split_half"),
    (1, 2, 1, 1, 128, True, 10000.0, "split_half"),
    (1, 4, 4, 257, 64, True, 500000.0, "split_half"),
    (1, 6, 2, 96, 128, False, 0.0, "split_half"),
    (1, 4, 2, 150, 128, True, 10000.0, "adjacent"),
    (2, 2, 2, 385, 64, True, 10000.0, "split_half"),
]


@pytest.mark.parametrize("B,hq,hkv,T,d,causal,base,layout", CASES)
def test_bwd_parity(B, hq, hkv, T, d, causal, base, layout):
    w = W.PrefillWorkload("bwd", B=B, Hq=hq, Hkv=hkv, T=T, d=d, dtype="bf16", rope_base=base,
                          scale=1.0 / math.sqrt(d), causal=causal, seed=T + d + hq)
    q, k, v = W.make_prefill_inputs(w)
    g = torch.Generator()
    g.manual_seed(T)
    do = torch.randn(B, hq, T, d, generator=g).to(torch.bfloat16)
    dq, dk, dv = _run(q, k, v, do, causal, base, layout, w.scale)
    rq, rk, rv = OA.attention_backward(q, k, v, do, causal=causal, rope_base=base, scale=w.scale,
                                       rope_layout=layout, operand_dtype="bf16")
    _close(to_np(dq), rq, "dq")
    _close(to_np(dk), rk, "dk")
    _close(to_np(dv), rv, "dv")


def test_bwd_llama_workload_one_group():
    """Full-size workload; one KV group (4 query heads) of one batch entry checked."""
    w = W.WORKLOADS["llama_gqa_bf16"]
    q, k, v = W.make_prefill_inputs(w)
    g = torch.Generator()
    g.manual_seed(99)
    do = torch.randn(w.B, w.Hq, w.T, w.d, generator=g).to(torch.bfloat16)
    dq, dk, dv = _run(q, k, v, do, True, w.rope_base, "split_half", w.scale)
    b, grp = 2, 5
    rep = w.Hq // w.Hkv
    hs = slice(grp * rep, (grp + 1) * rep)
    rq, rk, rv = OA.attention_backward(q[b:b + 1, hs], k[b:b + 1, grp:grp + 1],
                                       v[b:b + 1, grp:grp + 1], do[b:b + 1, hs], causal=True,
                                       rope_base=w.rope_base, scale=w.scale, operand_dtype="bf16")
    _close(to_np(dq[b:b + 1, hs]), rq, "dq group")
    _close(to_np(dk[b:b + 1, grp:grp + 1]), rk, "dk group")
    _close(to_np(dv[b:b + 1, grp:grp + 1]), rv, "dv group")


@pytest.mark.parametrize("B,hq,hkv,T,d,causal", [
    (4, 48, 16, 512, 64, False),    # 768 dQ work items: several per persistent CTA
    (4, 64, 64, 300, 128, True),    # MHA, odd query-tile count
])
def test_bwd_many_items_per_cta(B, hq, hkv, T, d, causal):
    """More work items than SMs, so the persistent dQ kernel reuses both TMEM
    accumulators; two KV groups checked against the oracle."""
    w = W.PrefillWorkload("bwd_many", B=B, Hq=hq, Hkv=hkv, T=T, d=d, dtype="bf16",
                          rope_base=10000.0, scale=1.0 / math.sqrt(d), causal=causal,
                          seed=B + hq + T)
    q, k, v = W.make_prefill_inputs(w)
    g = torch.Generator()
    g.manual_seed(T + 1)
    do = torch.randn(B, hq, T, d, generator=g).to(torch.bfloat16)
    dq, dk, dv = _run(q, k, v, do, causal, w.rope_base, "split_half", w.scale)
    rep = hq // hkv
    for b, grp in [(0, hkv - 1), (3, hkv // 2)]:
        hs = slice(grp * rep, (grp + 1) * rep)
        rq, rk, rv = OA.attention_backward(q[b:b + 1, hs], k[b:b + 1, grp:grp + 1],
                                           v[b:b + 1, grp:grp + 1], do[b:b + 1, hs],
                                           causal=causal, rope_base=w.rope_base, scale=w.scale,
                                           operand_dtype="bf16")
        _close(to_np(dq[b:b + 1, hs]), rq, f"dq ({b},{grp})")
        _close(to_np(dk[b:b + 1, grp:grp + 1]), rk, f"dk ({b},{grp})")
        _close(to_np(dv[b:b + 1, grp:grp + 1]), rv, f"dv ({b},{grp})")


def test_bwd_gqa_equals_summed_mha():
    """dk, dv of a GQA group equal the sums over its heads of the MHA gradients on repeated
    K/V (the group sum the kernel does in registers)."""
    B, Hq, Hkv, T, d = 1, 4, 1, 150, 128
    w = W.PrefillWorkload("g", B=B, Hq=Hq, Hkv=Hkv, T=T, d=d, dtype="bf16", rope_base=10000.0,
                          scale=1.0 / math.sqrt(d), seed=7)
    q, k, v = W.make_prefill_inputs(w)
    g = torch.Generator()
    g.manual_seed(8)
    do = torch.randn(B, Hq, T, d, generator=g).to(torch.bfloat16)
    dq, dk, dv = _run(q, k, v, do, True, w.rope_base, "split_half", w.scale)
    dq2, dk2, dv2 = _run(q, k.repeat_interleave(Hq, 1).contiguous(),
                         v.repeat_interleave(Hq, 1).contiguous(), do, True, w.rope_base,
                         "split_half", w.scale)
    _close(to_np(dq), to_np(dq2), "dq gqa vs mha")
    _close(to_np(dk), to_np(dk2).sum(axis=1, keepdims=True), "dk gqa vs summed mha")
    _close(to_np(dv), to_np(dv2).sum(axis=1, keepdims=True), "dv gqa vs summed mha")


# ------------------------------------------------------------------ fp32 (SIMT)
# fp32 operands, fp32 arithmetic throughout (accurate sine/cosine for RoPE, fp32
# forward out and lse): each gradient entry is a sum of at most T products of
# terms carrying a few fp32 roundings (2^-24 ~ 6e-8) each, and P = exp(S - lse)
# carries the absolute error of S and lse (~1e-6 for |S| ~ 10).  Bound: the
# fp32 parity bound, max-abs 1e-5 (absolute), and relative L2 1e-5; the relative L2 floor
# is 0.1 sqrt(n) (RMS error <= 1e-6 where the exact gradient vanishes, T = 1).

FP32_CASES = [
    # (B, Hq, Hkv, T, d, causal, rope_base, layout)
    (2, 4, 2, 97, 16, True, 10000.0, "split_half"),
    (1, 2, 2, 1, 16, False, 0.0, "split_half"),
    (2, 6, 2, 130, 32, True, 10000.0, "adjacent"),
    (1, 4, 1, 200, 32, False, 500000.0, "split_half"),
    (2, 4, 2, 150, 64, True, 10000.0, "split_half"),
    (1, 3, 3, 65, 64, False, 0.0, "split_half"),
    (1, 4, 1, 1, 128, True, 10000.0, "split_half"),
    (2, 4, 2, 129, 128, True, 10000.0, "adjacent"),
    (1, 8, 2, 77, 128, False, 10000.0, "split_half"),
]


@pytest.mark.parametrize("B,hq,hkv,T,d,causal,base,layout", FP32_CASES)
def test_bwd_fp32_parity(B, hq, hkv, T, d, causal, base, layout):
    w = W.PrefillWorkload("bwd32", B=B, Hq=hq, Hkv=hkv, T=T, d=d, dtype="f32", rope_base=base,
                          scale=1.0 / math.sqrt(d), causal=causal, seed=3 * T + d + hq)
    q, k, v = W.make_prefill_inputs(w)
    g = torch.Generator()
    g.manual_seed(T + 1)
    do = torch.randn(B, hq, T, d, generator=g, dtype=torch.float32)
    dq, dk, dv = _run(q, k, v, do, causal, base, layout, w.scale)
    assert dq.dtype == torch.float32 and dk.dtype == torch.float32
    rq, rk, rv = OA.attention_backward(q, k, v, do, causal=causal, rope_base=base, scale=w.scale,
                                       rope_layout=layout, operand_dtype="f32")
    tol = dict(rl2_tol=1e-5, abs_tol=1e-5, floor=0.1, bf16_storage=False)
    _close(to_np(dq), rq, "dq", **tol)
    _close(to_np(dk), rk, "dk", **tol)
    _close(to_np(dv), rv, "dv", **tol)
