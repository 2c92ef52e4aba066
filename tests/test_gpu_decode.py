"""Decode parity and the failure-detection paths, through the C ABI."""
import math

import numpy as np
import pytest
import torch

import attn_workloads as W
import transformer_causal_self_gb300 as csattn
from oracle import attn as OA
from tests.gpu_helpers import assert_bf16_close, assert_f32_close, dev, to_np

pytestmark = pytest.mark.gpu


def _decode(q, kc, vc, lens, **kw):
    out = csattn.attn_decode(q.to(dev()), kc.to(dev()), vc.to(dev()), lens.to(dev()), **kw)
    csattn.check_status()
    return out


def test_decode_workload_full():
    w = W.WORKLOADS["decode_bf16"]
    q, kc, vc, lens = W.make_decode_inputs(w)
    out = _decode(q, kc, vc, lens, scale=w.scale, max_seq_len=int(lens.max()))
    ref = OA.decode(q, kc, vc, lens.numpy(), scale=w.scale)
    assert_bf16_close(to_np(out), ref, "decode")


@pytest.mark.parametrize("Hq,Hkv,d", [(8, 8, 128), (16, 4, 128), (16, 2, 64), (32, 2, 128), (6, 2, 64)])
def test_decode_groups_and_lengths(Hq, Hkv, d):
    lens = [1, 63, 64, 65, 128, 1000, 777]
    w = W.DecodeWorkload("dec", B=len(lens), Hq=Hq, Hkv=Hkv, d=d, Lmax=1000, Lmin=1,
                         scale=1.0 / math.sqrt(d), seed=Hq + d)
    q, kc, vc, sl = W.make_decode_inputs(w, seq_lens=lens)
    ref = OA.decode(q, kc, vc, sl.numpy(), scale=w.scale)
    for splits in (0, 1, 3, 16):
        out = _decode(q, kc, vc, sl, scale=w.scale, max_seq_len=1000, num_splits=splits)
        assert_bf16_close(to_np(out), ref, f"decode splits={splits}")


def test_decode_split_count_invariance():
    """Results agree across split counts within bf16 rounding.

    Each split rounds its P = 2^(x - m_s) to bf16 against its own running max
    m_s, so two split counts see independent P rounding: about 2^-9/sqrt(3)
    relative noise per weight, which reaches the output at ~1e-3 relative and
    at sqrt(2) times that between two runs.  The bound is therefore the bf16
    parity bound (max-abs 2e-2, rel-L2 5e-3), and each result is also held to
    the oracle.
    """
    w = W.WORKLOADS["decode_bf16"].with_(B=8, Lmax=4096, Lmin=512)
    q, kc, vc, sl = W.make_decode_inputs(w)
    ref = OA.decode(q, kc, vc, sl.numpy(), scale=w.scale)
    outs = [to_np(_decode(q, kc, vc, sl, scale=w.scale, max_seq_len=4096, num_splits=s))
            for s in (1, 4, 7, 64)]
    for s, o in zip((1, 4, 7, 64), outs):
        assert_bf16_close(o, ref, f"splits={s}")
        err = np.max(np.abs(o - outs[0]))
        rl2 = np.linalg.norm(o - outs[0]) / np.linalg.norm(outs[0])
        assert err <= 2e-2 and rl2 <= 5e-3, (s, err, rl2)


def test_decode_matches_prefill_last_row():
    """Decode at length L equals row L-1 of the prefill on the same rotated data."""
    T, d = 700, 128
    w = W.WORKLOADS["llama_gqa_bf16"].with_(B=2, Hq=8, Hkv=2, T=T)
    q, k, v = W.make_prefill_inputs(w)
    full = csattn.attn_fwd(q.to(dev()), k.to(dev()), v.to(dev()), causal=True,
                           rope_base=w.rope_base, scale=w.scale).cpu()
    # pre-rotated query and cache as the oracle rounds them (inputs, not expected values)
    qr = torch.from_numpy(OA.round_to_bf16(OA.rope_rotate(q.double().numpy(), np.arange(T),
                                                          w.rope_base))).to(torch.bfloat16)
    kr = torch.from_numpy(OA.round_to_bf16(OA.rope_rotate(k.double().numpy(), np.arange(T),
                                                          w.rope_base))).to(torch.bfloat16)
    lens = torch.tensor([T, 311], dtype=torch.int32)
    qd = torch.stack([qr[0, :, T - 1:T], qr[1, :, 310:311]]).contiguous()
    out = _decode(qd, kr.contiguous(), v, lens, scale=w.scale, max_seq_len=T).cpu()
    assert_bf16_close(to_np(out[0, :, 0]), to_np(full[0, :, T - 1]), "decode vs prefill row")
    ref = OA.decode(qd, kr, v, lens.numpy(), scale=w.scale)
    assert_bf16_close(to_np(out), ref, "decode vs oracle")


def test_decode_bad_seq_len_sets_device_error():
    w = W.WORKLOADS["decode_bf16"].with_(B=3, Lmax=256, Lmin=1)
    q, kc, vc, _ = W.make_decode_inputs(w, seq_lens=[10, 20, 30])
    lens = torch.tensor([10, 0, 30], dtype=torch.int32)
    out = csattn.attn_decode(q.to(dev()), kc.to(dev()), vc.to(dev()), lens.to(dev()),
                             scale=w.scale, max_seq_len=256)
    with pytest.raises(csattn.CsattnError) as e:
        csattn.check_status()
    assert e.value.status == -6
    assert torch.all(out[1].float().cpu() == 0)
    csattn.check_status()  # cleared


def test_bounded_wait_reports_timeout_and_context_survives():
    csattn.selftest_bounded_wait(2000)
    with pytest.raises(csattn.CsattnError) as e:
        csattn.check_status()
    assert e.value.status == -4
    csattn.check_status()  # cleared, context usable
    w = W.WORKLOADS["llama_gqa_bf16"].with_(B=1, Hq=2, Hkv=1, T=130)
    q, k, v = W.make_prefill_inputs(w)
    out = csattn.attn_fwd(q.to(dev()), k.to(dev()), v.to(dev()), rope_base=w.rope_base,
                          scale=w.scale)
    csattn.check_status()
    ref = OA.attention(q, k, v, causal=True, rope_base=w.rope_base, scale=w.scale,
                       operand_dtype="bf16")
    assert_bf16_close(to_np(out), ref, "after timeout")


@pytest.mark.parametrize("Hq,Hkv,d,dv", [(16, 4, 128, 64), (8, 2, 64, 128), (32, 2, 64, 128),
                                          (6, 6, 128, 64)])
def test_decode_value_width_differs(Hq, Hkv, d, dv):
    """csattn_attn_decode_ext: keys d wide, values and output dv wide ("Transformer Math
    and Implementation Deep Dive", "Attention Equation"), against the oracle over ragged
    lengths (NaN past each sequence's rows) and several split counts."""
    lens = [1, 63, 64, 65, 300, 1000, 777]
    B, Lmax = len(lens), 1000
    g = torch.Generator()
    g.manual_seed(Hq + d + 3 * dv)
    q = torch.randn(B, Hq, 1, d, generator=g).to(torch.bfloat16)
    kc = torch.full((B, Hkv, Lmax, d), float("nan")).to(torch.bfloat16)
    vc = torch.full((B, Hkv, Lmax, dv), float("nan")).to(torch.bfloat16)
    for b, L in enumerate(lens):
        kc[b, :, :L] = torch.randn(Hkv, L, d, generator=g).to(torch.bfloat16)
        vc[b, :, :L] = torch.randn(Hkv, L, dv, generator=g).to(torch.bfloat16)
    sl = torch.tensor(lens, dtype=torch.int32)
    ref = OA.decode(q, kc, vc, sl.numpy())
    for splits in (0, 1, 5):
        out = csattn.attn_decode_ext(q.to(dev()), kc.to(dev()), vc.to(dev()), sl.to(dev()),
                                     max_seq_len=Lmax, num_splits=splits)
        csattn.check_status()
        assert out.shape == (B, Hq, 1, dv)
        assert_bf16_close(to_np(out), ref, f"decode_ext d={d} dv={dv} splits={splits}")


def test_decode_ext_equal_widths_is_decode():
    """dv = d through csattn_attn_decode_ext runs the same kernels as csattn_attn_decode:
    the outputs are equal bit for bit."""
    w = W.WORKLOADS["decode_bf16"].with_(B=6, Lmax=2048, Lmin=1)
    q, kc, vc, sl = (t.to(dev()) for t in W.make_decode_inputs(w))
    sl = sl.to(torch.int32)
    a = csattn.attn_decode(q, kc, vc, sl, scale=w.scale, max_seq_len=2048)
    b = csattn.attn_decode_ext(q, kc, vc, sl, scale=w.scale, max_seq_len=2048)
    csattn.check_status()
    assert torch.equal(a, b)


@pytest.mark.parametrize("Hq,Hkv,d", [(8, 2, 128), (4, 4, 64), (12, 3, 32), (2, 1, 16),
                                      (40, 2, 64)])
def test_decode_fp32_parity(Hq, Hkv, d):
    """fp32 decode (SIMT, fp32 throughout) against the oracle at the fp32 parity bound
    (max-abs 1e-5), ragged lengths with NaN past each sequence's rows, several split
    counts; the group of 20 query heads is past the bf16 kernels' limit of 16."""
    lens = [1, 31, 32, 33, 300, 777, 1000]
    w = W.DecodeWorkload("dec32", B=len(lens), Hq=Hq, Hkv=Hkv, d=d, Lmax=1000, Lmin=1,
                         dtype="f32", scale=1.0 / math.sqrt(d), seed=Hq + d)
    q, kc, vc, sl = W.make_decode_inputs(w, seq_lens=lens)
    assert q.dtype == torch.float32
    ref = OA.decode(q, kc, vc, sl.numpy(), scale=w.scale)
    for splits in (0, 1, 3, 16):
        out = _decode(q, kc, vc, sl, scale=w.scale, max_seq_len=1000, num_splits=splits)
        assert out.dtype == torch.float32
        assert_f32_close(to_np(out), ref, f"fp32 decode splits={splits}")


def test_decode_fp32_rows_equal_prefill_rows():
    """The incremental decode reproduces the one-shot forward ("The Transformer
    architecture", "Hands-on": in fp32 the two agree to a few 1e-7): decoding query t
    over keys 0..t gives row t of the fp32 causal prefill on the same K and V."""
    B, Hq, Hkv, T, d = 2, 8, 2, 300, 64
    g = torch.Generator()
    g.manual_seed(123)
    q = torch.randn(B, Hq, T, d, generator=g)
    k = torch.randn(B, Hkv, T, d, generator=g)
    v = torch.randn(B, Hkv, T, d, generator=g)
    pre = csattn.attn_fwd(q.to(dev()), k.to(dev()), v.to(dev()), causal=True, rope_base=0.0)
    csattn.check_status()
    worst = 0.0
    for t in (0, 1, 127, 128, 200, T - 1):
        lens = torch.full((B,), t + 1, dtype=torch.int32)
        out = _decode(q[:, :, t:t + 1].contiguous(), k, v, lens, max_seq_len=T)
        worst = max(worst, float((out[:, :, 0] - pre[:, :, t]).abs().max()))
    assert worst <= 1e-6, worst


@pytest.mark.parametrize("layout", ["split_half", "adjacent"])
def test_decode_fp32_generation_with_rope(layout):
    """An fp32 generation loop through the library alone: the RoPE pass in fp32 builds the
    rotated queries and key cache (checked against the oracle's rotation), and decoding
    query t over keys 0..t reproduces row t of the fp32 prefill with RoPE."""
    B, Hq, Hkv, T, d, base = 2, 4, 2, 200, 32, 10000.0
    g = torch.Generator()
    g.manual_seed(77)
    q = torch.randn(B, Hq, T, d, generator=g)
    k = torch.randn(B, Hkv, T, d, generator=g)
    v = torch.randn(B, Hkv, T, d, generator=g)
    qd, kd, vd = q.to(dev()), k.to(dev()), v.to(dev())
    pre = csattn.attn_fwd(qd, kd, vd, causal=True, rope_base=base, rope_layout=layout)
    q_rot = csattn.rope_rotate(qd, rope_base=base, rope_layout=layout)
    k_rot = csattn.rope_rotate(kd, rope_base=base, rope_layout=layout)
    csattn.check_status()
    ref_k = OA.rope_rotate(k.double().numpy(), np.arange(T), base, layout)
    assert np.max(np.abs(to_np(k_rot) - ref_k)) < 2e-6
    worst = 0.0
    for t in (0, 63, 64, 150, T - 1):
        lens = torch.full((B,), t + 1, dtype=torch.int32)
        out = _decode(q_rot[:, :, t:t + 1].contiguous(), k_rot, vd, lens, max_seq_len=T)
        worst = max(worst, float((out[:, :, 0] - pre[:, :, t]).abs().max()))
    assert worst <= 2e-6, worst
