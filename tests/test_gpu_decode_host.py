"""KV-cache decode from host buffers (csattn_attn_decode_host): only the rows below
seq_lens are copied (every other cache row holds NaN on the host and is never
copied), and the result equals the device decode bit for bit with one chunk and the
float64 oracle within the usual tolerance with several."""
import numpy as np
import pytest
import torch

import attn_workloads as W
import transformer_causal_self_gb300 as csattn
from oracle import attn as OA
from tests.gpu_helpers import assert_bf16_close, dev

pytestmark = pytest.mark.gpu


def _inputs(B, Hq, Hkv, Lmax, d, seed):
    w = W.WORKLOADS["decode_bf16"].with_(B=B, Hq=Hq, Hkv=Hkv, Lmax=Lmax, d=d)
    g = torch.Generator()
    g.manual_seed(seed)
    q = torch.randn(B, Hq, 1, d, generator=g).to(torch.bfloat16)
    kc = torch.randn(B, Hkv, Lmax, d, generator=g).to(torch.bfloat16)
    vc = torch.randn(B, Hkv, Lmax, d, generator=g).to(torch.bfloat16)
    lens = torch.randint(1, Lmax + 1, (B,), generator=g, dtype=torch.int32)
    lens[0] = Lmax
    lens[-1] = 1
    for b in range(B):
        kc[b, :, int(lens[b]):] = float("nan")
        vc[b, :, int(lens[b]):] = float("nan")
    return w, q, kc, vc, lens


@pytest.mark.parametrize("B,Hq,Hkv,Lmax,d,chunks,splits", [
    (6, 8, 2, 1000, 128, 0, 0),
    (5, 4, 4, 300, 64, 3, 2),
    (16, 32, 8, 2048, 128, 16, 0),
])
def test_decode_host_parity(B, Hq, Hkv, Lmax, d, chunks, splits):
    w, q, kc, vc, lens = _inputs(B, Hq, Hkv, Lmax, d, seed=B + Lmax)
    out = csattn.attn_decode_host(q.pin_memory(), kc.pin_memory(), vc.pin_memory(), lens,
                                  scale=w.scale, num_splits=splits, num_chunks=chunks)
    torch.cuda.synchronize()
    csattn.check_status()
    ref = OA.decode(q, kc, vc, lens.tolist(), scale=w.scale)
    assert_bf16_close(out.float().numpy(), ref, "host decode")


def test_decode_host_one_chunk_bit_exact_with_device_call():
    w, q, kc, vc, lens = _inputs(7, 16, 4, 700, 128, seed=3)
    out_h = csattn.attn_decode_host(q.pin_memory(), kc.pin_memory(), vc.pin_memory(), lens,
                                    scale=w.scale, num_chunks=1)
    torch.cuda.synchronize()
    out_d = csattn.attn_decode(q.to(dev()), kc.to(dev()), vc.to(dev()), lens.to(dev()),
                               scale=w.scale, max_seq_len=int(lens.max()))
    csattn.check_status()
    assert torch.equal(out_h, out_d.cpu())


def test_decode_host_rejects_bad_length_on_the_host():
    w, q, kc, vc, lens = _inputs(3, 4, 2, 64, 64, seed=4)
    lens[1] = 65
    with pytest.raises(csattn.CsattnError) as e:
        csattn.attn_decode_host(q, kc, vc, lens, scale=w.scale)
    assert e.value.status == -1
    assert np.all(np.isfinite(q.float().numpy()))
