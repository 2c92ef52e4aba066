"""Chunked prefill over a paged KV cache (csattn_attn_prefill_paged) against the
float64 oracle (oracle.attn.prefill_paged) on the same bf16 inputs, and against the
contiguous chunked prefill (csattn_attn_fwd_ext) on the same rows.

The page pools are built on the host: keys rotated and rounded to bf16 by the
oracle's rotation, placed into shuffled pages; every cache row at or past a
sequence's end holds NaN, which the kernel must never let into the output."""
import math

import numpy as np
import pytest
import torch

import attn_workloads as W
import transformer_causal_self_gb300 as csattn
from oracle import attn as OA
from tests.gpu_helpers import assert_bf16_close, dev, to_np

pytestmark = pytest.mark.gpu


def _g(seed):
    g = torch.Generator()
    g.manual_seed(seed)
    return g


def _paged_inputs(B, Hq, Hkv, Tq, d, page, lens, base, layout, seed, spare=2):
    """q [B,Hq,Tq,d]; pools of rotated keys and values with rows 0..lens[b]+Tq-1 per
    sequence (NaN past them); the contiguous rotated caches they were cut from."""
    g = _g(seed)
    Lmax = max(lens) + Tq
    Lmax = -(-Lmax // page) * page
    q = torch.randn(B, Hq, Tq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(B, Hkv, Lmax, d, generator=g, dtype=torch.float64)
    v = torch.randn(B, Hkv, Lmax, d, generator=g).to(torch.bfloat16)
    if base > 0:
        kr = OA.round_to_bf16(OA.rope_rotate(k.numpy(), np.arange(Lmax), base, layout))
        kr = torch.from_numpy(kr).to(torch.bfloat16)
    else:
        kr = k.to(torch.bfloat16)
    for b, L in enumerate(lens):
        kr[b, :, L + Tq:] = float("nan")
        v[b, :, L + Tq:] = float("nan")
    ends = [L + Tq for L in lens]
    kp, vp, table = W.page_cache(kr, v, ends, page, seed=seed, spare=spare)
    return q, kr, v, kp, vp, table


CASES = [
    # (B, Hq, Hkv, Tq, page, lens, rope_base, layout, causal)
    (3, 8, 2, 200, 128, [0, 77, 300], 10000.0, "split_half", True),
    (2, 4, 4, 130, 64, [64, 191], 10000.0, "adjacent", True),
    (2, 6, 2, 64, 192, [5, 400], 0.0, "split_half", True),
    (1, 2, 1, 1, 256, [1000], 10000.0, "split_half", True),
    (2, 4, 2, 100, 128, [30, 129], 500000.0, "split_half", False),
    (4, 32, 8, 256, 256, [0, 511, 1024, 1777], 10000.0, "split_half", True),
    (2, 3, 1, 300, 64, [17, 0], 10000.0, "split_half", True),
    (2, 4, 2, 150, 16, [33, 200], 10000.0, "split_half", True),   # 16-row pages
    (2, 8, 2, 97, 32, [0, 131], 10000.0, "adjacent", False),      # 32-row pages
]


@pytest.mark.parametrize("B,Hq,Hkv,Tq,page,lens,base,layout,causal", CASES)
def test_prefill_paged_parity(B, Hq, Hkv, Tq, page, lens, base, layout, causal):
    d = 128
    q, _, _, kp, vp, table = _paged_inputs(B, Hq, Hkv, Tq, d, page, lens, base, layout,
                                           seed=Tq + page + sum(lens))
    lens_d = torch.tensor(lens, dtype=torch.int32, device=dev())
    lse = torch.empty(B, Hq, Tq, dtype=torch.float32, device=dev())
    out = csattn.attn_prefill_paged(q.to(dev()), kp.to(dev()), vp.to(dev()), table.to(dev()),
                                    lens_d, causal=causal, rope_base=base, rope_layout=layout,
                                    scale=1.0 / math.sqrt(d), lse=lse)
    csattn.check_status()
    ref, ref_lse = OA.prefill_paged(q, kp.double().numpy(), vp.double().numpy(), table.numpy(),
                                    lens, page, causal=causal, rope_base=base, rope_layout=layout,
                                    scale=1.0 / math.sqrt(d), operand_dtype="bf16", lse=True)
    assert_bf16_close(to_np(out), ref, "paged prefill")
    assert np.max(np.abs(to_np(lse) - ref_lse)) < 2e-2


D64_CASES = [
    # (B, Hq, Hkv, Tq, page, lens, rope_base, layout, causal): head size 64
    (2, 4, 4, 200, 64, [0, 150], 10000.0, "split_half", True),
    (3, 12, 12, 129, 128, [77, 0, 300], 0.0, "split_half", True),
    (2, 8, 2, 64, 192, [5, 250], 10000.0, "adjacent", False),
    (1, 6, 2, 1, 64, [500], 10000.0, "split_half", True),
    (2, 4, 2, 130, 16, [70, 3], 10000.0, "split_half", True),
]


@pytest.mark.parametrize("B,Hq,Hkv,Tq,page,lens,base,layout,causal", D64_CASES)
def test_prefill_paged_parity_d64(B, Hq, Hkv, Tq, page, lens, base, layout, causal):
    d = 64
    q, _, _, kp, vp, table = _paged_inputs(B, Hq, Hkv, Tq, d, page, lens, base, layout,
                                           seed=3 * Tq + page + sum(lens))
    lens_d = torch.tensor(lens, dtype=torch.int32, device=dev())
    lse = torch.empty(B, Hq, Tq, dtype=torch.float32, device=dev())
    out = csattn.attn_prefill_paged(q.to(dev()), kp.to(dev()), vp.to(dev()), table.to(dev()),
                                    lens_d, causal=causal, rope_base=base, rope_layout=layout,
                                    scale=1.0 / math.sqrt(d), lse=lse)
    csattn.check_status()
    ref, ref_lse = OA.prefill_paged(q, kp.double().numpy(), vp.double().numpy(), table.numpy(),
                                    lens, page, causal=causal, rope_base=base, rope_layout=layout,
                                    scale=1.0 / math.sqrt(d), operand_dtype="bf16", lse=True)
    assert_bf16_close(to_np(out), ref, "paged prefill d=64")
    assert np.max(np.abs(to_np(lse) - ref_lse)) < 2e-2


@pytest.mark.parametrize("page,d", [(64, 128), (128, 128), (384, 128), (64, 64), (256, 64),
                                    (16, 128), (32, 64)])
def test_prefill_paged_bit_exact_with_contiguous_chunk(page, d):
    """Same rows in pages and in a contiguous cache: the paged chunk equals the
    contiguous chunked prefill (keys given rotated) bit for bit."""
    B, Hq, Hkv, Tq, L = 2, 8, 2, 300, 229
    q, kr, v, kp, vp, table = _paged_inputs(B, Hq, Hkv, Tq, d, page, [L, L], 10000.0,
                                            "split_half", seed=page + d)
    lens_d = torch.tensor([L, L], dtype=torch.int32, device=dev())
    out_p = csattn.attn_prefill_paged(q.to(dev()), kp.to(dev()), vp.to(dev()), table.to(dev()),
                                      lens_d, rope_base=10000.0)
    kc = kr[:, :, :L + Tq].contiguous().to(dev())
    vc = v[:, :, :L + Tq].contiguous().to(dev())
    out_c = csattn.attn_fwd_ext(q.to(dev()), kc, vc, q_offset=L, rope_base=10000.0,
                                k_prerotated=True)
    csattn.check_status()
    assert torch.equal(out_p, out_c), float((out_p.float() - out_c.float()).abs().max())


@pytest.mark.parametrize("page", [128, 16])
def test_prefill_paged_bad_page_and_length_set_device_error(page):
    B, Hq, Hkv, Tq, d = 3, 4, 2, 100, 128
    lens = [50, 200, 10]
    q, _, _, kp, vp, table = _paged_inputs(B, Hq, Hkv, Tq, d, page, lens, 0.0, "split_half",
                                           seed=11)
    table[1, 1] = kp.shape[0]  # one past the pool, inside sequence 1's rows
    qd, kpd, vpd = q.to(dev()), kp.to(dev()), vp.to(dev())
    out = csattn.attn_prefill_paged(qd, kpd, vpd, table.to(dev()),
                                    torch.tensor(lens, dtype=torch.int32, device=dev()))
    with pytest.raises(csattn.CsattnError) as e:
        csattn.check_status()
    assert e.value.status == -6
    for b in (0, 2):  # the other sequences are unaffected
        ref = OA.prefill_paged(q[b:b + 1], kp.double().numpy(), vp.double().numpy(),
                               table[b:b + 1].numpy(), [lens[b]], page, operand_dtype="bf16")
        assert_bf16_close(to_np(out[b:b + 1]), ref, f"sequence {b}")
    csattn.check_status()  # cleared
    # a length past the logical cache: reported, nothing read out of bounds
    bad = torch.tensor([50, table.shape[1] * page, 10], dtype=torch.int32, device=dev())
    csattn.attn_prefill_paged(qd, kpd, vpd, table.to(dev()), bad)
    with pytest.raises(csattn.CsattnError) as e:
        csattn.check_status()
    assert e.value.status == -6
    csattn.check_status()


def test_prefill_paged_chunk_workload_sampled_rows():
    """The bench's paged row at full size: llama_chunk_bf16 (1024 queries after 3072
    cached rows) with the rotated cache in 256-row pages of a shuffled pool; sampled
    rows of three heads against the contiguous definition."""
    w = W.WORKLOADS["llama_chunk_bf16"]
    q, k, v = W.make_chunk_inputs(w)
    kr = OA.round_to_bf16(OA.rope_rotate(k.double().numpy(), np.arange(w.Tk), w.rope_base))
    kp, vp, table = W.page_cache(torch.from_numpy(kr).to(torch.bfloat16), v, [w.Tk] * w.B, 256,
                                 seed=21, spare=3)
    lens = torch.full((w.B,), w.q_offset, dtype=torch.int32, device=dev())
    out = csattn.attn_prefill_paged(q.to(dev()), kp.to(dev()), vp.to(dev()), table.to(dev()),
                                    lens, rope_base=w.rope_base, scale=w.scale)
    csattn.check_status()
    oc = out.cpu()
    for b, h in ((0, 5), (2, 18), (3, 31)):
        rows = W.sample_query_rows(w.Tq, 96, seed=b * 100 + h + 7)
        ref = OA.attention_rows(q, k, v, b, h, rows, causal=True, rope_base=w.rope_base,
                                scale=w.scale, operand_dtype="bf16", q_offset=w.q_offset)
        assert_bf16_close(oc[b, h, rows].double().numpy(), ref, f"paged chunk b={b} h={h}")
