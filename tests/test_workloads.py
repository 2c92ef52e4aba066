"""The seeded input generators and the work counts the bench divides by."""
import random

import attn_workloads as W


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
