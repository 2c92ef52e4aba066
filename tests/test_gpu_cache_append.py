"""Appending a chunk of tokens to contiguous and paged KV caches (csattn_cache_append,
csattn_cache_append_paged) against the float64 oracle, and the caches it leaves in
use: a paged decode and a chunked prefill over the appended rows."""
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


def _bits(t):
    return t.contiguous().view(torch.int16).cpu()


def _check_rows(got_k, got_v, want_k, want_v, written):
    """Written rows: values bit-exact, rotated keys equal to the oracle's rounding in all but
    rare last-bit ties; every other row bit-identical to what was there."""
    gk, gv = got_k.double().numpy(), got_v.double().numpy()
    m = written
    assert np.array_equal(gv[m], want_v[m])
    match = np.mean(gk[m] == want_k[m])
    assert match >= 0.999, match
    assert np.max(np.abs(gk[m] - want_k[m])) <= 2.0 ** -7 * np.max(np.abs(want_k[m]))
    keep = ~m
    both_nan = np.isnan(gk[keep]) & np.isnan(want_k[keep])
    assert np.all((gk[keep] == want_k[keep]) | both_nan)
    both_nan = np.isnan(gv[keep]) & np.isnan(want_v[keep])
    assert np.all((gv[keep] == want_v[keep]) | both_nan)


@pytest.mark.parametrize("d,Hkv,Tn,base,layout", [
    (128, 8, 300, 10000.0, "split_half"),
    (64, 2, 1, 500000.0, "adjacent"),
    (128, 4, 17, 0.0, "split_half"),
])
def test_cache_append_contiguous(d, Hkv, Tn, base, layout):
    B, Lmax = 3, 1024
    lens = [0, 257, Lmax - Tn]
    g = _g(d + Tn)
    kn = torch.randn(B, Hkv, Tn, d, generator=g).to(torch.bfloat16)
    vn = torch.randn(B, Hkv, Tn, d, generator=g).to(torch.bfloat16)
    kc = torch.full((B, Hkv, Lmax, d), float("nan"), dtype=torch.bfloat16)
    vc = torch.full((B, Hkv, Lmax, d), float("nan"), dtype=torch.bfloat16)
    kc_d, vc_d = kc.to(dev()), vc.to(dev())
    csattn.cache_append(kn.to(dev()), vn.to(dev()), kc_d, vc_d,
                        torch.tensor(lens, dtype=torch.int32, device=dev()), rope_base=base,
                        rope_layout=layout)
    csattn.check_status()
    wk, wv = OA.cache_append(kn, vn, kc, vc, lens, rope_base=base, rope_layout=layout,
                             operand_dtype="bf16")
    written = np.zeros(wk.shape, dtype=bool)
    for b, L in enumerate(lens):
        written[b, :, L:L + Tn] = True
    _check_rows(kc_d.cpu(), vc_d.cpu(), wk, wv, written)


@pytest.mark.parametrize("page", [128, 16])
def test_cache_append_paged_then_decode(page):
    """A 1024-token prompt appended in three chunks into shuffled pages, then a paged
    decode over ragged prefixes of it equals the oracle's decode over the same pages."""
    B, Hq, Hkv, d = 3, 16, 4, 128
    n_lp = 1024 // page
    g = _g(11)
    k = torch.randn(B, Hkv, 1024, d, generator=g).to(torch.bfloat16)
    v = torch.randn(B, Hkv, 1024, d, generator=g).to(torch.bfloat16)
    q = torch.randn(B, Hq, 1, d, generator=g).to(torch.bfloat16)
    n_pages = B * n_lp + 2
    table = torch.randperm(n_pages, generator=g)[:B * n_lp].to(torch.int32).view(B, n_lp)
    table = table.contiguous()
    table_d = table.to(dev())
    kp = torch.full((n_pages, Hkv, page, d), float("nan"), dtype=torch.bfloat16, device=dev())
    vp = torch.full((n_pages, Hkv, page, d), float("nan"), dtype=torch.bfloat16, device=dev())
    kp_ref = np.full((n_pages, Hkv, page, d), np.nan)
    vp_ref = np.full((n_pages, Hkv, page, d), np.nan)
    L = 0
    for Tn in (200, 300, 524):
        kn, vn = k[:, :, L:L + Tn].contiguous(), v[:, :, L:L + Tn].contiguous()
        lens = [L] * B
        csattn.cache_append_paged(kn.to(dev()), vn.to(dev()), kp, vp, table_d,
                                  torch.tensor(lens, dtype=torch.int32, device=dev()),
                                  rope_base=10000.0)
        csattn.check_status()
        kp_ref, vp_ref = OA.cache_append_paged(kn, vn, kp_ref, vp_ref, table.numpy(), lens, page,
                                               rope_base=10000.0, operand_dtype="bf16")
        L += Tn
    # the pages hold what the oracle's paged append wrote (keys up to rare last-bit ties)
    _check_rows(kp.cpu(), vp.cpu(), kp_ref, vp_ref, ~np.isnan(kp_ref))
    lens = [300, 777, 1024]
    out = csattn.attn_decode_paged(q.to(dev()), kp, vp, table_d,
                                   torch.tensor(lens, dtype=torch.int32, device=dev()))
    csattn.check_status()
    ref = OA.decode_paged(q, kp_ref, vp_ref, table.numpy(), lens, page)
    assert_bf16_close(to_np(out), ref, "paged decode after append")


def test_append_then_chunked_prefill_matches_full_prefill():
    """A prompt's first 768 tokens appended to a cache, then a 256-query chunk over the
    cache plus the chunk's own appended keys reproduces the last rows of a full prefill."""
    w = W.WORKLOADS["llama_gqa_bf16"].with_(B=2, Hq=8, Hkv=2, T=1024)
    q, k, v = W.make_prefill_inputs(w)
    kc = torch.zeros(2, 2, 1024, 128, dtype=torch.bfloat16, device=dev())
    vc = torch.zeros_like(kc)
    zero = torch.zeros(2, dtype=torch.int32, device=dev())
    csattn.cache_append(k.to(dev()), v.to(dev()), kc, vc, zero, rope_base=w.rope_base)
    out = csattn.attn_fwd_ext(q[:, :, 768:].contiguous().to(dev()), kc, vc, q_offset=768,
                              causal=True, rope_base=w.rope_base, scale=w.scale,
                              k_prerotated=True)
    csattn.check_status()
    full = csattn.attn_fwd(q.to(dev()), k.to(dev()), v.to(dev()), causal=True,
                           rope_base=w.rope_base, scale=w.scale)
    assert torch.equal(out.view(torch.int16), full[:, :, 768:].contiguous().view(torch.int16))


def test_cache_append_out_of_range_sets_device_error():
    B, Hkv, Tn, d, Lmax = 2, 2, 8, 64, 64
    kn = torch.randn(B, Hkv, Tn, d).to(torch.bfloat16).to(dev())
    vn = torch.randn(B, Hkv, Tn, d).to(torch.bfloat16).to(dev())
    kc = torch.zeros(B, Hkv, Lmax, d, dtype=torch.bfloat16, device=dev())
    vc = torch.zeros_like(kc)
    bad = torch.tensor([3, Lmax - Tn + 1], dtype=torch.int32, device=dev())
    csattn.cache_append(kn, vn, kc, vc, bad, rope_base=10000.0)
    with pytest.raises(csattn.CsattnError) as e:
        csattn.check_status()
    assert e.value.status == -6
    assert torch.all(kc[1] == 0) and torch.all(vc[1] == 0)   # the bad sequence untouched
    assert torch.equal(vc[0, :, 3:3 + Tn].cpu(), vn[0].cpu())  # the good one written
    csattn.check_status()  # cleared
