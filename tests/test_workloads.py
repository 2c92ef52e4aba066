"""The seeded input generators and the work counts the bench divides by."""
import random

import numpy as np
import torch

import attn_workloads as W
from oracle import attn as OA


def test_chunk_visible_keys_brute_force():
    r = random.Random(1)
    for _ in range(2000):
        w = W.ChunkWorkload("t", 1, 1, 1, r.randint(1, 60), r.randint(1, 60), r.randint(0, 80), 8,
                            "f32", 0.0, 1.0, r.random() < 0.8)
        brute = sum(min(w.Tk, w.q_offset + i + 1) if w.causal else w.Tk for i in range(w.Tq))
        assert w.visible_keys() == brute


def test_chunk_workload_shapes_and_flops():
    w = W.WORKLOADS["llama_chunk_bf16"]
    assert w.Tk == w.q_offset + w.Tq
    q, k, v = W.make_chunk_inputs(w.with_(B=1, Hq=4, Hkv=1))
    assert q.shape == (1, 4, w.Tq, w.d) and k.shape == (1, 1, w.Tk, w.d) == v.shape
    # rows 0..1023 see 3073..4096 keys
    assert w.visible_keys() == sum(range(3073, 4097))
    assert w.flops() == 4.0 * w.B * w.Hq * w.d * w.visible_keys()


def test_page_cache_places_every_row():
    """The page scatter is pure placement: gathering back through the table gives the
    contiguous rows, and the oracle's paged decode equals its contiguous decode."""
    g = torch.Generator().manual_seed(11)
    kc = torch.randn(3, 2, 200, 8, generator=g).to(torch.bfloat16)
    vc = torch.randn(3, 2, 200, 8, generator=g).to(torch.bfloat16)
    q = torch.randn(3, 4, 1, 8, generator=g).to(torch.bfloat16)
    lens = [1, 64, 200]
    kp, vp, table = W.page_cache(kc, vc, lens, 64, seed=3, spare=2)
    assert kp.shape == (1 + 1 + 4 + 2, 2, 64, 8) and table.shape == (3, 4)
    for b, L in enumerate(lens):
        for t in range(L):
            assert torch.equal(kp[table[b, t // 64], :, t % 64], kc[b, :, t])
            assert torch.equal(vp[table[b, t // 64], :, t % 64], vc[b, :, t])
        assert torch.all(table[b, -(-L // 64):] == -1)
    used = table[table >= 0]
    assert len(set(used.tolist())) == used.numel()
    got = OA.decode_paged(q, kp.double().numpy(), vp.double().numpy(), table.numpy(), lens, 64)
    assert np.max(np.abs(got - OA.decode(q, kc.double().numpy(), vc.double().numpy(), lens))) == 0
