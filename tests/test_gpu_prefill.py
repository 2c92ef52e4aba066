"""Prefill parity: the CUDA path (through the C ABI) against the float64 oracle."""
import math

import numpy as np
import pytest
import torch

import attn_workloads as W
import transformer_causal_self_gb300 as csattn
from oracle import attn as OA
from tests.gpu_helpers import assert_bf16_close, assert_f32_close, dev, to_np

pytestmark = pytest.mark.gpu


def _run(q, k, v, **kw):
    out = csattn.attn_fwd(q.to(dev()), k.to(dev()), v.to(dev()), **kw)
    csattn.check_status()
    return out


# ------------------------------------------------------------------ fp32 (SIMT)

@pytest.mark.parametrize("layout", ["split_half", "adjacent"])
def test_tiny_fp32_workload(layout):
    w = W.WORKLOADS["tiny_f32"].with_(rope_layout=layout)
    q, k, v = W.make_prefill_inputs(w)
    out = _run(q, k, v, causal=True, rope_base=w.rope_base, scale=w.scale, rope_layout=layout)
    ref = OA.attention(q, k, v, causal=True, rope_base=w.rope_base, scale=w.scale,
                       rope_layout=layout, operand_dtype="f32")
    assert_f32_close(to_np(out), ref, f"tiny fp32 {layout}")


FP32_CASES = [
    # (d, Hq, Hkv, T, causal)
    (16, 2, 2, 1, True), (16, 4, 1, 37, True), (16, 6, 2, 200, False),
    (32, 2, 2, 37, True), (32, 6, 2, 200, True), (32, 4, 1, 1, False),
    (64, 4, 1, 200, True), (64, 2, 2, 37, False), (64, 6, 2, 129, True),
    (128, 2, 2, 200, True), (128, 6, 2, 37, False), (128, 4, 1, 1, True),
    (128, 4, 4, 97, True),
]


@pytest.mark.parametrize("d,hq,hkv,T,causal", FP32_CASES)
def test_fp32_shapes(d, hq, hkv, T, causal):
    base = 10000.0 if (d + T) % 2 == 0 else 0.0
    w = W.PrefillWorkload("f32case", B=2, Hq=hq, Hkv=hkv, T=T, d=d, dtype="f32", rope_base=base,
                          scale=1.0 / math.sqrt(d), causal=causal, seed=d + T)
    q, k, v = W.make_prefill_inputs(w)
    lse = torch.empty(2, hq, T, dtype=torch.float32, device=dev())
    out = _run(q, k, v, causal=causal, rope_base=base, scale=w.scale, lse=lse)
    ref = OA.attention(q, k, v, causal=causal, rope_base=base, scale=w.scale, operand_dtype="f32")
    assert_f32_close(to_np(out), ref, "fp32 shapes")
    ref_lse = OA.attention_lse(q, k, causal=causal, rope_base=base, scale=w.scale, operand_dtype="f32")
    assert np.max(np.abs(to_np(lse) - ref_lse)) < 1e-4


# ------------------------------------------------------------------ bf16 (tcgen05)

BF16_CASES = [
    # (B, Hq, Hkv, T, d, causal, rope_base, layout)
    (1, 2, 1, 1, 128, True, 10000.0, "split_half"),
    (1, 2, 1, 127, 128, True, 10000.0, "split_half"),
    (1, 4, 1, 128, 128, True, 10000.0, "adjacent"),
    (2, 4, 2, 129, 128, True, 0.0, "split_half"),
    (1, 8, 2, 300, 128, True, 500000.0, "split_half"),
    (1, 4, 4, 513, 128, True, 10000.0, "split_half"),   # MHA: consecutive-tile units, odd tile count
    (1, 3, 1, 385, 128, True, 10000.0, "adjacent"),     # odd group: head pair + consecutive tiles
    (2, 2, 2, 256, 64, True, 0.0, "split_half"),
    (1, 6, 2, 700, 64, True, 10000.0, "split_half"),
    (1, 4, 1, 333, 128, False, 10000.0, "split_half"),  # no mask
    (1, 2, 2, 200, 64, False, 0.0, "split_half"),
    (3, 2, 1, 1000, 128, True, 10000.0, "split_half"),
]


@pytest.mark.parametrize("B,Hq,Hkv,T,d,causal,base,layout", BF16_CASES)
def test_bf16_parity(B, Hq, Hkv, T, d, causal, base, layout):
    w = W.PrefillWorkload("bf16case", B=B, Hq=Hq, Hkv=Hkv, T=T, d=d, dtype="bf16", rope_base=base,
                          scale=1.0 / math.sqrt(d), causal=causal, seed=T + 7 * d + Hq,
                          rope_layout=layout)
    q, k, v = W.make_prefill_inputs(w)
    out = torch.full((B, Hq, T, d), float("nan"), dtype=torch.bfloat16, device=dev())
    lse = torch.full((B, Hq, T), float("nan"), dtype=torch.float32, device=dev())
    _run(q, k, v, out=out, causal=causal, rope_base=base, scale=w.scale, rope_layout=layout, lse=lse)
    ref = OA.attention(q, k, v, causal=causal, rope_base=base, scale=w.scale, rope_layout=layout,
                       operand_dtype="bf16")
    assert_bf16_close(to_np(out), ref, f"bf16 {B},{Hq},{Hkv},{T},{d}")
    ref_lse = OA.attention_lse(q, k, causal=causal, rope_base=base, scale=w.scale,
                               rope_layout=layout, operand_dtype="bf16")
    assert np.max(np.abs(to_np(lse) - ref_lse)) < 2e-2


@pytest.mark.parametrize("B,Hq,Hkv,T,d", [
    (4, 64, 64, 300, 128),   # MHA, 3 query tiles: the longest units have no tile A
    (4, 48, 16, 300, 128),   # group of 3: head pairs, then consecutive-tile units
    (4, 64, 64, 300, 64),
])
def test_bf16_many_units_per_cta(B, Hq, Hkv, T, d):
    """Enough units that every CTA runs several, among them the single-tile units of
    an odd tile count ahead of two-tile ones; a sample of heads against the oracle."""
    w = W.PrefillWorkload("many_units", B=B, Hq=Hq, Hkv=Hkv, T=T, d=d, dtype="bf16",
                          rope_base=10000.0, scale=1.0 / math.sqrt(d), causal=True,
                          seed=B + Hq + d)
    q, k, v = W.make_prefill_inputs(w)
    out = _run(q, k, v, causal=True, rope_base=w.rope_base, scale=w.scale).cpu()
    rep = Hq // Hkv
    for b, h in [(0, 0), (1, Hq - 1), (2, Hq // 2 + 1), (3, 7), (3, Hq - 2)]:
        g = h // rep
        ref = OA.attention(q[b:b + 1, h:h + 1], k[b:b + 1, g:g + 1], v[b:b + 1, g:g + 1],
                           causal=True, rope_base=w.rope_base, scale=w.scale,
                           operand_dtype="bf16")
        assert_bf16_close(to_np(out[b:b + 1, h:h + 1]), ref, f"head ({b},{h})")


def test_bf16_rotated_keys_match_oracle_rounding():
    """The rotated keys (left in the workspace) equal the oracle's rounded rotation."""
    w = W.WORKLOADS["llama_gqa_bf16"].with_(B=1, Hq=4, Hkv=2, T=1000)
    q, k, v = W.make_prefill_inputs(w)
    ws = torch.empty(csattn.fwd_workspace_size(1, 4, 2, 1000, 128, torch.bfloat16, w.rope_base),
                     dtype=torch.uint8, device=dev())
    _run(q, k, v, causal=True, rope_base=w.rope_base, scale=w.scale, workspace=ws)
    k_rot = ws.view(torch.bfloat16).view(1, 2, 1000, 128)
    ref = OA.round_to_bf16(OA.rope_rotate(k.double().numpy(), np.arange(1000), w.rope_base))
    match = np.mean(to_np(k_rot) == ref)
    assert match >= 0.999, match
    assert np.max(np.abs(to_np(k_rot) - ref)) <= 2 ** -7 * np.max(np.abs(ref))


def test_causality_bit_exact():
    """Changing q/k/v at position j leaves every output row i < j bit-identical."""
    w = W.WORKLOADS["llama_gqa_bf16"].with_(B=1, Hq=4, Hkv=1, T=640)
    q, k, v = W.make_prefill_inputs(w)
    base = _run(q, k, v, causal=True, rope_base=w.rope_base, scale=w.scale).cpu()
    for j in (9, 128, 383, 639):
        q2, k2, v2 = q.clone(), k.clone(), v.clone()
        q2[:, :, j] += 3.0
        k2[:, :, j] -= 2.0
        v2[:, :, j] *= -5.0
        got = _run(q2, k2, v2, causal=True, rope_base=w.rope_base, scale=w.scale).cpu()
        assert torch.equal(got[:, :, :j], base[:, :, :j]), j
        assert not torch.equal(got[:, :, j], base[:, :, j])


def test_gqa_equals_mha_with_repeated_kv():
    w = W.WORKLOADS["llama_gqa_bf16"].with_(B=2, Hq=8, Hkv=2, T=300)
    q, k, v = W.make_prefill_inputs(w)
    a = _run(q, k, v, causal=True, rope_base=w.rope_base, scale=w.scale).cpu()
    kr = k.repeat_interleave(4, dim=1).contiguous()
    vr = v.repeat_interleave(4, dim=1).contiguous()
    b = _run(q, kr, vr, causal=True, rope_base=w.rope_base, scale=w.scale).cpu()
    # the same kernel on the same bytes: each query row's arithmetic does not depend on
    # which KV head number its keys carry or which tile it is paired with
    assert torch.equal(a, b), (a.float() - b.float()).abs().max().item()


def test_gpt2_workload_full():
    w = W.WORKLOADS["gpt2_bf16"]
    q, k, v = W.make_prefill_inputs(w)
    out = _run(q, k, v, causal=True, rope_base=0.0, scale=w.scale)
    ref = OA.attention(q, k, v, causal=True, rope_base=0.0, scale=w.scale, operand_dtype="bf16")
    assert_bf16_close(to_np(out), ref, "gpt2")


def _sampled(w, heads, n_rows, full_head=None):
    q, k, v = W.make_prefill_inputs(w)
    out = _run(q, k, v, causal=True, rope_base=w.rope_base, scale=w.scale).cpu()
    got_all, ref_all = [], []
    for (b, h) in heads:
        rows = W.sample_query_rows(w.T, n_rows, seed=b * 131 + h)
        ref = OA.attention_rows(q, k, v, b, h, rows, causal=True, rope_base=w.rope_base,
                                scale=w.scale, operand_dtype="bf16")
        got_all.append(out[b, h, rows].double().numpy())
        ref_all.append(ref)
    if full_head is not None:
        b, h = full_head
        rows = np.arange(w.T)
        ref = OA.attention_rows(q, k, v, b, h, rows, causal=True, rope_base=w.rope_base,
                                scale=w.scale, operand_dtype="bf16")
        got_all.append(out[b, h].double().numpy())
        ref_all.append(ref)
    return np.concatenate(got_all), np.concatenate(ref_all)


@pytest.mark.parametrize("name", ["llama_gqa_bf16", "llama_gqa_bf16_x4"])
def test_llama_workload_sampled(name):
    w = W.WORKLOADS[name]
    got, ref = _sampled(w, heads=[(0, 1), (1, 14), (2, 31), (3, 7)], n_rows=256,
                        full_head=(0, 0))
    assert_bf16_close(got, ref, name)


def test_long_workload_sampled():
    w = W.WORKLOADS["long_gqa_bf16"]
    got, ref = _sampled(w, heads=[(0, 0), (0, 13), (0, 30)], n_rows=400)
    assert_bf16_close(got, ref, "long")


# ------------------------------------------------------------------ largest sizes

def test_bf16_at_the_largest_rope_position():
    """T = 49152, the longest sequence RoPE accepts (positions up to 49151, angles up to
    49151 rad for the first channel pair): sampled rows, the last row included."""
    w = W.PrefillWorkload("maxpos", B=1, Hq=2, Hkv=1, T=49152, d=128, dtype="bf16",
                          rope_base=10000.0, scale=1.0 / math.sqrt(128), seed=17)
    got, ref = _sampled(w, heads=[(0, 0), (0, 1)], n_rows=96)
    assert_bf16_close(got, ref, "T=49152")


def test_fp32_at_the_largest_rope_position():
    w = W.PrefillWorkload("maxpos32", B=1, Hq=2, Hkv=1, T=49152, d=16, dtype="f32",
                          rope_base=10000.0, scale=0.25, causal=True, seed=18)
    q, k, v = W.make_prefill_inputs(w)
    out = _run(q, k, v, causal=True, rope_base=w.rope_base, scale=w.scale).cpu()
    for h in (0, 1):
        rows = W.sample_query_rows(w.T, 64, seed=h + 3)
        ref = OA.attention_rows(q, k, v, 0, h, rows, causal=True, rope_base=w.rope_base,
                                scale=w.scale, operand_dtype="f32")
        assert_f32_close(out[0, h, rows].double().numpy(), ref, f"fp32 T=49152 h={h}")
