"""Chunked prefill (queries at an offset after a cache prefix) and rectangular
attention through csattn_attn_fwd_ext, against the float64 oracle."""
import math

import numpy as np
import pytest
import torch

import attn_workloads as W
import transformer_causal_self_gb300 as csattn
from oracle import attn as OA
from tests.gpu_helpers import assert_bf16_close, assert_f32_close, dev, to_np

pytestmark = pytest.mark.gpu


def _inputs(B, Hq, Hkv, Tq, Tk, d, dtype, seed):
    w = W.ChunkWorkload("case", B=B, Hq=Hq, Hkv=Hkv, Tq=Tq, Tk=Tk, q_offset=0, d=d, dtype=dtype,
                        rope_base=0.0, scale=0.0, seed=seed)
    return W.make_chunk_inputs(w)


def _run(q, k, v, **kw):
    out = csattn.attn_fwd_ext(q.to(dev()), k.to(dev()), v.to(dev()), **kw)
    csattn.check_status()
    return out


F32_CASES = [
    # (d, Hq, Hkv, Tq, Tk, q_offset, causal, rope_base)
    (16, 4, 1, 16, 64, 48, True, 10000.0),
    (32, 2, 2, 33, 70, 37, True, 10000.0),
    (64, 6, 2, 20, 45, 0, False, 0.0),
    (128, 4, 4, 1, 300, 299, True, 10000.0),
    (64, 4, 2, 50, 40, 30, True, 10000.0),    # rows past the last key see every key
    (16, 2, 1, 70, 9, 5, False, 10000.0),
]


@pytest.mark.parametrize("d,hq,hkv,Tq,Tk,off,causal,base", F32_CASES)
def test_fp32_chunks(d, hq, hkv, Tq, Tk, off, causal, base):
    q, k, v = _inputs(2, hq, hkv, Tq, Tk, d, "f32", seed=d + Tq + Tk)
    lse = torch.empty(2, hq, Tq, dtype=torch.float32, device=dev())
    out = _run(q, k, v, q_offset=off, causal=causal, rope_base=base, scale=0.0, lse=lse)
    ref = OA.attention(q, k, v, causal=causal, rope_base=base, operand_dtype="f32", q_offset=off)
    assert_f32_close(to_np(out), ref, "fp32 chunk")
    ref_lse = OA.attention_lse(q, k, causal=causal, rope_base=base, operand_dtype="f32",
                               q_offset=off)
    assert np.max(np.abs(to_np(lse) - ref_lse)) < 1e-4


BF16_CASES = [
    # (d, Hq, Hkv, Tq, Tk, q_offset, causal, rope_base)
    (128, 8, 2, 128, 512, 384, True, 10000.0),   # aligned chunk, head pairs
    (128, 8, 2, 200, 700, 500, True, 10000.0),   # ragged chunk and offset
    (128, 3, 3, 257, 1000, 743, True, 10000.0),  # odd group: consecutive tiles
    (128, 4, 1, 1, 300, 299, True, 10000.0),     # one query (decode-shaped)
    (128, 4, 2, 300, 129, 0, False, 0.0),        # rectangular, Tq > Tk
    (128, 4, 2, 77, 513, 10, False, 10000.0),    # rectangular with RoPE at an offset
    (128, 4, 2, 150, 100, 60, True, 10000.0),    # rows past the last key
    (64, 8, 2, 200, 700, 500, True, 10000.0),
    (64, 6, 6, 129, 300, 0, False, 0.0),
    (64, 4, 1, 1, 1, 0, True, 10000.0),
]


@pytest.mark.parametrize("d,hq,hkv,Tq,Tk,off,causal,base", BF16_CASES)
def test_bf16_chunks(d, hq, hkv, Tq, Tk, off, causal, base):
    q, k, v = _inputs(2, hq, hkv, Tq, Tk, d, "bf16", seed=3 * d + Tq + Tk)
    lse = torch.empty(2, hq, Tq, dtype=torch.float32, device=dev())
    out = torch.full((2, hq, Tq, d), float("nan"), dtype=torch.bfloat16, device=dev())
    _run(q, k, v, out=out, q_offset=off, causal=causal, rope_base=base, scale=0.0, lse=lse)
    ref = OA.attention(q, k, v, causal=causal, rope_base=base, operand_dtype="bf16", q_offset=off)
    assert_bf16_close(to_np(out), ref, "bf16 chunk")
    ref_lse = OA.attention_lse(q, k, causal=causal, rope_base=base, operand_dtype="bf16",
                               q_offset=off)
    assert np.max(np.abs(to_np(lse) - ref_lse)) < 2e-3


@pytest.mark.parametrize("d,hq,hkv,Tq,Tk,off,causal", [
    (128, 64, 64, 300, 1000, 700, True),    # MHA, odd query-tile count at an offset
    (128, 48, 16, 300, 500, 0, False),      # group of 3, rectangular
    (64, 64, 64, 300, 800, 500, True),
])
def test_bf16_chunks_many_units_per_cta(d, hq, hkv, Tq, Tk, off, causal):
    """More units than SMs (several per CTA, single-tile units among them); a sample of
    heads against the oracle."""
    B = 4
    q, k, v = _inputs(B, hq, hkv, Tq, Tk, d, "bf16", seed=d + hq + Tq)
    out = _run(q, k, v, q_offset=off, causal=causal, rope_base=10000.0, scale=0.0).cpu()
    rep = hq // hkv
    for b, h in [(0, 0), (1, hq - 1), (2, hq // 2 + 1), (3, 5)]:
        g = h // rep
        ref = OA.attention(q[b:b + 1, h:h + 1], k[b:b + 1, g:g + 1], v[b:b + 1, g:g + 1],
                           causal=causal, rope_base=10000.0, operand_dtype="bf16", q_offset=off)
        assert_bf16_close(to_np(out[b:b + 1, h:h + 1]), ref, f"head ({b},{h})")


@pytest.mark.parametrize("d", [64, 128])
def test_aligned_chunks_reproduce_full_prefill_bitwise(d):
    """Chunks at offsets that are multiples of the 128-row tile run the same tiles in
    the same order as the full prefill: their rows match it bit for bit."""
    w = W.PrefillWorkload("full", B=2, Hq=8, Hkv=2, T=1024, d=d, dtype="bf16",
                          rope_base=10000.0, scale=1.0 / math.sqrt(d), seed=21)
    q, k, v = (t.to(dev()) for t in W.make_prefill_inputs(w))
    full = csattn.attn_fwd(q, k, v, causal=True, rope_base=w.rope_base, scale=w.scale)
    for off, Tq in ((0, 256), (256, 384), (640, 384)):
        chunk = csattn.attn_fwd_ext(q[:, :, off:off + Tq].contiguous(), k[:, :, :off + Tq].contiguous(),
                                    v[:, :, :off + Tq].contiguous(), q_offset=off, causal=True,
                                    rope_base=w.rope_base, scale=w.scale)
        csattn.check_status()
        assert torch.equal(chunk, full[:, :, off:off + Tq]), off


def test_ragged_chunk_matches_full_prefill_rows():
    w = W.PrefillWorkload("full", B=1, Hq=8, Hkv=2, T=777, d=128, dtype="bf16",
                          rope_base=10000.0, scale=1.0 / math.sqrt(128), seed=22)
    q, k, v = (t.to(dev()) for t in W.make_prefill_inputs(w))
    full = csattn.attn_fwd(q, k, v, causal=True, rope_base=w.rope_base, scale=w.scale)
    off, Tq = 333, 300
    chunk = csattn.attn_fwd_ext(q[:, :, off:off + Tq].contiguous(), k[:, :, :off + Tq].contiguous(),
                                v[:, :, :off + Tq].contiguous(), q_offset=off, causal=True,
                                rope_base=w.rope_base, scale=w.scale)
    csattn.check_status()
    assert_bf16_close(to_np(chunk), to_np(full[:, :, off:off + Tq]), "ragged chunk vs full")


def test_single_query_chunk_matches_decode():
    """A one-query chunk at offset L-1 over pre-rotated keys is a decode step."""
    L, d = 1000, 128
    q, k, v = _inputs(3, 8, 2, 1, L, d, "bf16", seed=23)
    qd, kd, vd = q.to(dev()), k.to(dev()), v.to(dev())
    chunk = csattn.attn_fwd_ext(qd, kd, vd, q_offset=L - 1, causal=True, rope_base=0.0)
    lens = torch.full((3,), L, dtype=torch.int32, device=dev())
    dec = csattn.attn_decode(qd, kd, vd, lens, max_seq_len=L)
    csattn.check_status()
    assert_bf16_close(to_np(chunk), to_np(dec), "chunk of one vs decode")


def test_chunk_workload_sampled_rows():
    w = W.WORKLOADS["llama_chunk_bf16"]
    q, k, v = W.make_chunk_inputs(w)
    out = csattn.attn_fwd_ext(q.to(dev()), k.to(dev()), v.to(dev()), q_offset=w.q_offset,
                              causal=True, rope_base=w.rope_base, scale=w.scale)
    csattn.check_status()
    oc = out.cpu()
    for b, h in ((0, 0), (1, 13), (3, 31)):
        rows = W.sample_query_rows(w.Tq, 96, seed=b * 100 + h)
        ref = OA.attention_rows(q, k, v, b, h, rows, causal=True, rope_base=w.rope_base,
                                scale=w.scale, operand_dtype="bf16", q_offset=w.q_offset)
        assert_bf16_close(oc[b, h, rows].double().numpy(), ref, f"chunk workload b={b} h={h}")


def test_cross_workload_sampled_rows():
    """The rectangular (unmasked, cross-attention shaped) bench workload, sampled rows."""
    w = W.WORKLOADS["llama_cross_bf16"]
    q, k, v = W.make_chunk_inputs(w)
    out = csattn.attn_fwd_ext(q.to(dev()), k.to(dev()), v.to(dev()), q_offset=0, causal=False,
                              rope_base=0.0, scale=w.scale)
    csattn.check_status()
    oc = out.cpu()
    for b, h in ((0, 3), (2, 17), (3, 30)):
        rows = W.sample_query_rows(w.Tq, 96, seed=b * 100 + h + 1)
        ref = OA.attention_rows(q, k, v, b, h, rows, causal=False, rope_base=0.0, scale=w.scale,
                                operand_dtype="bf16")
        assert_bf16_close(oc[b, h, rows].double().numpy(), ref, f"cross workload b={b} h={h}")


@pytest.mark.parametrize("dtype,d,dv,hq,hkv,Tq,Tk,off,causal,base", [
    ("bf16", 64, 128, 8, 2, 200, 700, 500, True, 10000.0),   # narrow q, k; wide v
    ("bf16", 128, 64, 8, 2, 200, 700, 500, True, 10000.0),   # wide q, k; narrow v
    ("bf16", 64, 128, 6, 6, 300, 129, 0, False, 0.0),        # rectangular
    ("bf16", 128, 64, 4, 1, 129, 1000, 10, False, 10000.0),
    ("bf16", 64, 128, 64, 64, 300, 300, 0, True, 10000.0),    # many units per CTA
    ("f32", 16, 32, 4, 1, 16, 64, 48, True, 10000.0),
    ("f32", 128, 16, 2, 2, 33, 70, 37, True, 10000.0),
    ("f32", 32, 128, 6, 2, 20, 45, 0, False, 0.0),
])
def test_value_width_differs_from_key_width(dtype, d, dv, hq, hkv, Tq, Tk, off, causal, base):
    """v and out with dv channels, q and k with d ("Scaled dot-product attention": the
    weights come from q and k; v sets the output width)."""
    B = 2
    g = torch.Generator()
    g.manual_seed(d + 3 * dv + Tq)
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    q = torch.randn(B, hq, Tq, d, generator=g).to(dt)
    k = torch.randn(B, hkv, Tk, d, generator=g).to(dt)
    v = torch.randn(B, hkv, Tk, dv, generator=g).to(dt)
    lse = torch.empty(B, hq, Tq, dtype=torch.float32, device=dev())
    out = _run(q, k, v, q_offset=off, causal=causal, rope_base=base, scale=0.0, lse=lse)
    assert out.shape == (B, hq, Tq, dv)
    od = "bf16" if dtype == "bf16" else "f32"
    ref = OA.attention(q, k, v, causal=causal, rope_base=base, operand_dtype=od, q_offset=off)
    if dtype == "bf16":
        assert_bf16_close(to_np(out), ref, f"d={d} dv={dv}")
    else:
        assert_f32_close(to_np(out), ref, f"d={d} dv={dv}")
    ref_lse = OA.attention_lse(q, k, causal=causal, rope_base=base, operand_dtype=od, q_offset=off)
    assert np.max(np.abs(to_np(lse) - ref_lse)) < (2e-3 if dtype == "bf16" else 1e-4)
