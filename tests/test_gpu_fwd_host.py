"""Prefill from host buffers (csattn_attn_fwd_host): the pipelined copies in, chunked
attention and copies out give csattn_attn_fwd's results bit for bit, and the
float64 oracle's within the usual tolerance."""
import math

import pytest
import torch

import attn_workloads as W
import transformer_causal_self_gb300 as csattn
from oracle import attn as OA
from tests.gpu_helpers import assert_bf16_close, assert_f32_close, dev

pytestmark = pytest.mark.gpu


CASES = [
    # (B, Hq, Hkv, T, d, dtype, rope_base, num_chunks)
    (2, 8, 2, 300, 128, "bf16", 10000.0, 0),
    (2, 8, 2, 300, 128, "bf16", 10000.0, 1),
    (2, 8, 2, 300, 128, "bf16", 10000.0, 3),
    (2, 8, 2, 300, 128, "bf16", 10000.0, 16),
    (3, 6, 2, 200, 64, "bf16", 0.0, 0),
    (1, 4, 2, 100, 32, "f32", 10000.0, 2),
]


@pytest.mark.parametrize("B,Hq,Hkv,T,d,dtype,base,chunks", CASES)
def test_fwd_host_bit_exact_with_device_call(B, Hq, Hkv, T, d, dtype, base, chunks):
    w = W.PrefillWorkload("host", B=B, Hq=Hq, Hkv=Hkv, T=T, d=d, dtype=dtype, rope_base=base,
                          scale=1.0 / math.sqrt(d), causal=True, seed=B + T + d + chunks)
    q, k, v = W.make_prefill_inputs(w)
    hq, hk, hv = q.pin_memory(), k.pin_memory(), v.pin_memory()
    hlse = torch.empty(B, Hq, T, dtype=torch.float32).pin_memory()
    out_h = csattn.attn_fwd_host(hq, hk, hv, rope_base=base, scale=w.scale, lse=hlse,
                                 num_chunks=chunks)
    torch.cuda.synchronize()
    csattn.check_status()
    lse_d = torch.empty(B, Hq, T, dtype=torch.float32, device=dev())
    out_d = csattn.attn_fwd(q.to(dev()), k.to(dev()), v.to(dev()), rope_base=base, scale=w.scale,
                            lse=lse_d)
    csattn.check_status()
    assert torch.equal(out_h, out_d.cpu())
    assert torch.equal(hlse, lse_d.cpu())


def test_fwd_host_matches_oracle_on_a_user_stream():
    w = W.WORKLOADS["llama_gqa_bf16"].with_(B=2, Hq=8, Hkv=2, T=257)
    q, k, v = W.make_prefill_inputs(w)
    s = torch.cuda.Stream()
    out = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    csattn.attn_fwd_host(q.pin_memory(), k.pin_memory(), v.pin_memory(), out,
                         rope_base=w.rope_base, scale=w.scale, stream=s)
    s.synchronize()
    csattn.check_status()
    ref = OA.attention(q, k, v, causal=True, rope_base=w.rope_base, scale=w.scale,
                       operand_dtype="bf16")
    assert_bf16_close(out.float().numpy(), ref, "host-buffer prefill")


def test_fwd_host_pageable_memory():
    """Pageable host tensors work too (the copies are then not asynchronous)."""
    w = W.PrefillWorkload("host32", B=1, Hq=2, Hkv=1, T=64, d=16, dtype="f32", rope_base=10000.0,
                          scale=0.25, causal=True, seed=5)
    q, k, v = W.make_prefill_inputs(w)
    out = torch.empty_like(q)
    csattn.attn_fwd_host(q, k, v, out, rope_base=w.rope_base, scale=w.scale)
    torch.cuda.synchronize()
    csattn.check_status()
    ref = OA.attention(q, k, v, causal=True, rope_base=w.rope_base, scale=w.scale,
                       operand_dtype="f32")
    assert_f32_close(out.numpy(), ref, "pageable fp32")
