"""Decode with the cache append fused in (csattn_attn_decode_step) against the
float64 oracle's decode_step, plus the cache rows it writes and leaves alone."""

import numpy as np
import pytest
import torch

import transformer_causal_self_gb300 as csattn
from oracle import attn as OA
from tests.gpu_helpers import assert_bf16_close, dev, to_np

pytestmark = pytest.mark.gpu


def _g(seed):
    g = torch.Generator()
    g.manual_seed(seed)
    return g


def _setup(B, Hq, Hkv, Lmax, d, lens, base, layout, seed):
    """Caches holding rotated keys for rows < lens[b] and NaN beyond; new-token inputs."""
    g = _g(seed)
    k_seq = torch.randn(B, Hkv, Lmax, d, generator=g).to(torch.bfloat16)
    v_seq = torch.randn(B, Hkv, Lmax, d, generator=g).to(torch.bfloat16)
    q_new = torch.randn(B, Hq, 1, d, generator=g).to(torch.bfloat16)
    k_new = torch.randn(B, Hkv, 1, d, generator=g).to(torch.bfloat16)
    v_new = torch.randn(B, Hkv, 1, d, generator=g).to(torch.bfloat16)
    kc = torch.full((B, Hkv, Lmax, d), float("nan"), dtype=torch.bfloat16)
    vc = torch.full((B, Hkv, Lmax, d), float("nan"), dtype=torch.bfloat16)
    for b, L in enumerate(lens):
        if L == 0:
            continue
        kr = k_seq[b, :, :L]
        if base > 0:
            kr = torch.from_numpy(OA.round_to_bf16(OA.rope_rotate(kr.double().numpy(), np.arange(L),
                                                                   base, layout))).to(torch.bfloat16)
        kc[b, :, :L] = kr
        vc[b, :, :L] = v_seq[b, :, :L]
    return q_new, k_new, v_new, kc, vc


def _bits(t):
    return t.contiguous().view(torch.int16).cpu()


@pytest.mark.parametrize("d,Hq,Hkv,base,layout", [
    (128, 8, 2, 10000.0, "split_half"),
    (128, 32, 8, 500000.0, "split_half"),
    (64, 6, 2, 10000.0, "adjacent"),
    (64, 4, 4, 0.0, "split_half"),
])
def test_decode_step_parity_and_cache_rows(d, Hq, Hkv, base, layout):
    B, Lmax = 6, 700
    lens = [0, 1, 127, 128, 450, Lmax - 1]
    q_new, k_new, v_new, kc, vc = _setup(B, Hq, Hkv, Lmax, d, lens, base, layout, seed=d + Hq)
    kc_d, vc_d = kc.to(dev()), vc.to(dev())
    lens_d = torch.tensor(lens, dtype=torch.int32, device=dev())
    out = csattn.attn_decode_step(q_new.to(dev()), k_new.to(dev()), v_new.to(dev()), kc_d, vc_d,
                                  lens_d, rope_base=base, rope_layout=layout)
    csattn.check_status()
    ref, kc_ref, vc_ref = OA.decode_step(q_new, k_new, v_new, kc, vc, lens, rope_base=base,
                                         rope_layout=layout, operand_dtype="bf16")
    assert_bf16_close(to_np(out), ref, "decode step")
    # rows other than the new one are untouched, bit for bit (NaN fill included)
    kb, vb, kb0, vb0 = _bits(kc_d), _bits(vc_d), _bits(kc), _bits(vc)
    for b, p in enumerate(lens):
        others = [r for r in range(Lmax) if r != p]
        assert torch.equal(kb[b, :, others], kb0[b, :, others])
        assert torch.equal(vb[b, :, others], vb0[b, :, others])
        assert torch.equal(vc_d[b, :, p].cpu(), v_new[b, :, 0])
    # the written keys: the oracle's rotated, rounded key (a rare last-bit tie may differ)
    got = torch.stack([kc_d[b, :, p].cpu() for b, p in enumerate(lens)]).double().numpy()
    want = np.stack([kc_ref[b, :, p] for b, p in enumerate(lens)])
    match = np.mean(got == want)
    assert match >= 0.999, match
    assert np.max(np.abs(got - want)) <= 2.0 ** -7 * np.max(np.abs(want))


def test_generation_loop_matches_prefill():
    """Eight steps of append-and-attend reproduce the last rows of a causal prefill over
    the same (unrotated) sequence."""
    B, Hq, Hkv, d, T, base = 2, 8, 2, 128, 300, 10000.0
    g = _g(5)
    q = torch.randn(B, Hq, T, d, generator=g).to(torch.bfloat16)
    k = torch.randn(B, Hkv, T, d, generator=g).to(torch.bfloat16)
    v = torch.randn(B, Hkv, T, d, generator=g).to(torch.bfloat16)
    full = csattn.attn_fwd(q.to(dev()), k.to(dev()), v.to(dev()), causal=True, rope_base=base)
    start = T - 8
    kc = torch.zeros(B, Hkv, T, d, dtype=torch.bfloat16, device=dev())
    vc = torch.zeros(B, Hkv, T, d, dtype=torch.bfloat16, device=dev())
    kc[:, :, :start] = csattn.rope_rotate(k[:, :, :start].contiguous().to(dev()), rope_base=base)
    vc[:, :, :start] = v[:, :, :start].to(dev())
    lens = torch.full((B,), start, dtype=torch.int32, device=dev())
    for t in range(start, T):
        out = csattn.attn_decode_step(q[:, :, t:t + 1].contiguous().to(dev()),
                                      k[:, :, t:t + 1].contiguous().to(dev()),
                                      v[:, :, t:t + 1].contiguous().to(dev()), kc, vc, lens,
                                      rope_base=base)
        csattn.check_status()
        assert_bf16_close(to_np(out[:, :, 0]), to_np(full[:, :, t]), f"step {t}")
        lens += 1
    ref = OA.attention_rows(q, k, v, 1, 5, [T - 1], causal=True, rope_base=base,
                            operand_dtype="bf16")
    assert_bf16_close(to_np(out[1, 5]), ref, "last step vs oracle")


def test_decode_step_position_out_of_range_sets_device_error():
    B, Hq, Hkv, Lmax, d = 3, 4, 2, 64, 64
    lens = [5, 10, 3]
    q_new, k_new, v_new, kc, vc = _setup(B, Hq, Hkv, Lmax, d, lens, 10000.0, "split_half", 9)
    kc_d, vc_d = kc.to(dev()), vc.to(dev())
    bad = torch.tensor([5, Lmax, 3], dtype=torch.int32, device=dev())
    out = csattn.attn_decode_step(q_new.to(dev()), k_new.to(dev()), v_new.to(dev()), kc_d, vc_d,
                                  bad, rope_base=10000.0)
    with pytest.raises(csattn.CsattnError) as e:
        csattn.check_status()
    assert e.value.status == -6
    assert torch.equal(_bits(kc_d[1]), _bits(kc[1])) and torch.equal(_bits(vc_d[1]), _bits(vc[1]))
    assert torch.all(out[1].float().cpu() == 0)
    csattn.check_status()  # cleared
