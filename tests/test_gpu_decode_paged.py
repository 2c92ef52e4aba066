"""Decode over a paged KV cache (csattn_attn_decode_paged) against the float64
oracle's decode_paged, bit-for-bit against the contiguous decode, and the
device-side report of a page index outside the pool."""
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


def _paged(B, Hq, Hkv, d, page, n_lp, lens, spare, seed):
    """A contiguous cache of n_lp logical pages per sequence scattered into a shuffled
    pool with `spare` extra pages; pool rows that hold no key are NaN, table entries
    past a sequence's last page are -1 (never read)."""
    g = _g(seed)
    Lmax = n_lp * page
    kc = torch.randn(B, Hkv, Lmax, d, generator=g).to(torch.bfloat16)
    vc = torch.randn(B, Hkv, Lmax, d, generator=g).to(torch.bfloat16)
    q = torch.randn(B, Hq, 1, d, generator=g).to(torch.bfloat16)
    for b, L in enumerate(lens):
        kc[b, :, L:] = float("nan")
        vc[b, :, L:] = float("nan")
    n_pages = B * n_lp + spare
    perm = torch.randperm(n_pages, generator=g)
    kp = torch.full((n_pages, Hkv, page, d), float("nan"), dtype=torch.bfloat16)
    vp = torch.full((n_pages, Hkv, page, d), float("nan"), dtype=torch.bfloat16)
    table = torch.full((B, n_lp), -1, dtype=torch.int32)
    for b, L in enumerate(lens):
        for lp in range((L + page - 1) // page):
            pp = int(perm[b * n_lp + lp])
            table[b, lp] = pp
            kp[pp] = kc[b, :, lp * page:(lp + 1) * page]
            vp[pp] = vc[b, :, lp * page:(lp + 1) * page]
    return q, kc, vc, kp, vp, table


@pytest.mark.parametrize("d,Hq,Hkv,page,n_lp", [
    (128, 8, 2, 64, 12),
    (128, 32, 8, 128, 6),
    (64, 6, 2, 256, 3),
    (128, 16, 1, 64, 20),
    (128, 8, 2, 16, 50),     # 16-row pages: four pages per 64-row tile
    (64, 4, 4, 32, 21),      # 32-row pages, a logical cache that ends mid-tile
])
def test_decode_paged_parity(d, Hq, Hkv, page, n_lp):
    B = 6
    Lmax = n_lp * page
    lens = [1, page - 1, page, page + 1, Lmax // 2 + 3, Lmax]
    q, kc, vc, kp, vp, table = _paged(B, Hq, Hkv, d, page, n_lp, lens, 5, seed=d + Hq + page)
    lens_d = torch.tensor(lens, dtype=torch.int32, device=dev())
    out = csattn.attn_decode_paged(q.to(dev()), kp.to(dev()), vp.to(dev()), table.to(dev()),
                                   lens_d)
    csattn.check_status()
    ref = OA.decode_paged(q, kp.double().numpy(), vp.double().numpy(), table.numpy(), lens, page)
    assert_bf16_close(to_np(out), ref, "paged decode")


@pytest.mark.parametrize("num_splits", [0, 1, 3, 7])
def test_decode_paged_bit_exact_with_contiguous(num_splits):
    """Same chunking, same tiles, same arithmetic: the paged read changes only addresses."""
    B, Hq, Hkv, d, page, n_lp = 5, 16, 4, 128, 128, 10
    lens = [17, 128, 640, 1000, 1280]
    q, kc, vc, kp, vp, table = _paged(B, Hq, Hkv, d, page, n_lp, lens, 3, seed=40 + num_splits)
    lens_d = torch.tensor(lens, dtype=torch.int32, device=dev())
    qd = q.to(dev())
    paged = csattn.attn_decode_paged(qd, kp.to(dev()), vp.to(dev()), table.to(dev()), lens_d,
                                     num_splits=num_splits)
    contig = csattn.attn_decode(qd, kc.to(dev()), vc.to(dev()), lens_d, num_splits=num_splits)
    csattn.check_status()
    assert torch.equal(paged.view(torch.int16), contig.view(torch.int16))


def test_decode_paged_shared_prefix_pages():
    """Two sequences whose tables point at the same leading pages (a shared prompt)."""
    B, Hq, Hkv, d, page = 2, 8, 2, 128, 64
    g = _g(77)
    kp = torch.randn(7, Hkv, page, d, generator=g).to(torch.bfloat16)
    vp = torch.randn(7, Hkv, page, d, generator=g).to(torch.bfloat16)
    q = torch.randn(B, Hq, 1, d, generator=g).to(torch.bfloat16)
    table = torch.tensor([[4, 1, 6, -1], [4, 1, 0, 2]], dtype=torch.int32)
    lens = [3 * page - 10, 4 * page]
    out = csattn.attn_decode_paged(q.to(dev()), kp.to(dev()), vp.to(dev()), table.to(dev()),
                                   torch.tensor(lens, dtype=torch.int32, device=dev()))
    csattn.check_status()
    ref = OA.decode_paged(q, kp.double().numpy(), vp.double().numpy(), table.numpy(), lens, page)
    assert_bf16_close(to_np(out), ref, "shared-prefix pages")


def test_decode_paged_bad_page_sets_device_error():
    B, Hq, Hkv, d, page, n_lp = 3, 4, 2, 64, 64, 4
    lens = [100, 200, 50]
    q, kc, vc, kp, vp, table = _paged(B, Hq, Hkv, d, page, n_lp, lens, 0, seed=3)
    table[1, 2] = kp.shape[0]  # one past the pool, inside sequence 1's rows
    lens_d = torch.tensor(lens, dtype=torch.int32, device=dev())
    out = csattn.attn_decode_paged(q.to(dev()), kp.to(dev()), vp.to(dev()), table.to(dev()),
                                   lens_d)
    with pytest.raises(csattn.CsattnError) as e:
        csattn.check_status()
    assert e.value.status == -6
    # the other sequences are unaffected
    for b in (0, 2):
        ref = OA.decode_paged(q[b:b + 1], kp.double().numpy(), vp.double().numpy(),
                              table[b:b + 1].numpy(), [lens[b]], page)
        assert_bf16_close(to_np(out[b:b + 1]), ref, f"sequence {b}")
    csattn.check_status()  # cleared
