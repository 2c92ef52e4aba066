"""Backward of chunked and rectangular attention (csattn_attn_bwd_ext) against the
float64 oracle's gradients (oracle.attn.attention_backward with q_offset).

The chunk cases have Tq queries at positions q_offset.. after a prefix, so a query
tile meets keys from before the chunk ("The Transformer architecture", "Hands-on":
the query at position p sees keys 0..p); the rectangular cases drop the mask and
let Tq, Tk and the value width dv differ from the key width d ("Transformer Math
and Implementation Deep Dive", "Attention Equation").  Tolerances are those of
tests/test_gpu_bwd.py (bf16: relative L2 5e-3, max-abs 2e-2 plus half an ulp of
the largest entry; fp32: 1e-5)."""
import pytest
import torch

import transformer_causal_self_gb300 as csattn
from oracle import attn as OA
from tests.gpu_helpers import assert_grad_close, dev, to_np

pytestmark = pytest.mark.gpu

F32_TOL = dict(rl2_tol=1e-5, abs_tol=1e-5, floor=0.1, bf16_storage=False)


def _inputs(B, hq, hkv, Tq, Tk, d, dv, dtype, seed):
    g = torch.Generator()
    g.manual_seed(seed)
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    q = torch.randn(B, hq, Tq, d, generator=g).to(dt)
    k = torch.randn(B, hkv, Tk, d, generator=g).to(dt)
    v = torch.randn(B, hkv, Tk, dv, generator=g).to(dt)
    do = torch.randn(B, hq, Tq, dv, generator=g).to(dt)
    return q, k, v, do


def _run(q, k, v, do, off, causal, base, layout):
    qd, kd, vd, dod = (t.to(dev()) for t in (q, k, v, do))
    B, hq, Tq, _ = q.shape
    lse = torch.empty(B, hq, Tq, dtype=torch.float32, device=dev())
    out = csattn.attn_fwd_ext(qd, kd, vd, q_offset=off, causal=causal, rope_base=base,
                              rope_layout=layout, lse=lse)
    grads = csattn.attn_bwd_ext(qd, kd, vd, out, dod, lse, q_offset=off, causal=causal,
                                rope_base=base, rope_layout=layout)
    csattn.check_status()
    return grads


def _check(q, k, v, do, off, causal, base, layout, dtype, tag):
    dq, dk, dv = _run(q, k, v, do, off, causal, base, layout)
    assert dq.shape == q.shape and dk.shape == k.shape and dv.shape == v.shape
    rq, rk, rv = OA.attention_backward(q, k, v, do, causal=causal, rope_base=base,
                                       rope_layout=layout, operand_dtype=dtype, q_offset=off)
    tol = {} if dtype == "bf16" else F32_TOL
    assert_grad_close(to_np(dq), rq, f"{tag} dq", **tol)
    assert_grad_close(to_np(dk), rk, f"{tag} dk", **tol)
    assert_grad_close(to_np(dv), rv, f"{tag} dv", **tol)
    return dq, dk, dv


BF16_CASES = [
    # (B, Hq, Hkv, Tq, Tk, q_offset, d, dv, causal, rope_base, layout)
    (1, 4, 2, 128, 384, 256, 128, 128, True, 10000.0, "split_half"),  # aligned chunk
    (2, 4, 1, 130, 230, 100, 64, 64, True, 10000.0, "adjacent"),      # ragged chunk and offset
    (1, 3, 3, 257, 1000, 743, 128, 128, True, 500000.0, "split_half"),
    (1, 4, 1, 1, 300, 299, 128, 128, True, 10000.0, "split_half"),    # one query
    (1, 2, 2, 64, 400, 64, 128, 128, True, 10000.0, "split_half"),    # keys no query sees
    (1, 4, 2, 150, 100, 60, 128, 128, True, 10000.0, "split_half"),  # rows past the last key
    (1, 4, 2, 100, 300, 0, 128, 128, False, 0.0, "split_half"),       # rectangular, Tk > Tq
    (1, 6, 2, 300, 129, 0, 64, 64, False, 10000.0, "split_half"),     # rectangular, Tq > Tk
    (1, 4, 2, 77, 513, 10, 128, 128, False, 10000.0, "adjacent"),     # RoPE at an offset, no mask
    (1, 4, 2, 150, 150, 0, 128, 64, True, 10000.0, "split_half"),     # dv < d
    (1, 2, 1, 200, 333, 133, 64, 128, True, 10000.0, "split_half"),   # dv > d, chunk
    (2, 6, 3, 77, 190, 0, 64, 128, False, 10000.0, "split_half"),     # dv > d, rectangular
    (1, 4, 4, 200, 700, 500, 128, 64, True, 10000.0, "adjacent"),     # dv < d, chunk
]


@pytest.mark.parametrize("B,hq,hkv,Tq,Tk,off,d,dv,causal,base,layout", BF16_CASES)
def test_bwd_ext_bf16(B, hq, hkv, Tq, Tk, off, d, dv, causal, base, layout):
    q, k, v, do = _inputs(B, hq, hkv, Tq, Tk, d, dv, "bf16", seed=Tq + 3 * Tk + off + d + dv)
    _, dk, dv_ = _check(q, k, v, do, off, causal, base, layout, "bf16", "bf16")
    if causal and Tk > off + Tq:  # keys after the last query's position get no gradient
        assert torch.count_nonzero(dk[:, :, off + Tq:]).item() == 0
        assert torch.count_nonzero(dv_[:, :, off + Tq:]).item() == 0


EDGE_CASES = [
    # (dtype, B, Hq, Hkv, Tq, Tk, q_offset, d, dv, causal, rope_base)
    ("bf16", 1, 2, 1, 300, 1, 0, 128, 128, False, 10000.0),       # one key, many queries
    ("bf16", 1, 2, 2, 1, 1, 0, 64, 128, True, 10000.0),           # one query, one key
    ("bf16", 1, 4, 1, 128, 640, 49024, 128, 128, True, 10000.0),  # last row at position 49151
    ("f32", 1, 2, 1, 1, 1, 0, 16, 16, True, 10000.0),
    ("f32", 1, 2, 2, 40, 1, 7, 32, 64, True, 10000.0),            # one key seen by every row
]


@pytest.mark.parametrize("dtype,B,hq,hkv,Tq,Tk,off,d,dv,causal,base", EDGE_CASES)
def test_bwd_ext_edges(dtype, B, hq, hkv, Tq, Tk, off, d, dv, causal, base):
    """Degenerate shapes and the largest RoPE position: a single key (every visible
    row puts all its weight on it, so dq is zero up to rounding), a single query and
    key, and queries at positions 49024..49151 (all 640 keys visible to each)."""
    q, k, v, do = _inputs(B, hq, hkv, Tq, Tk, d, dv, dtype, seed=Tq + Tk + d + dv + 11)
    if Tk > 1:
        _check(q, k, v, do, off, causal, base, "split_half", dtype, f"edge {dtype}")
        return
    # one key: dS = P (dP - D) with P = 1 and dP = D exactly, so the exact dq and dk are
    # zero and only rounding of the two dot products remains (a relative L2 against zero
    # means nothing): max-abs for dq and dk, the full bounds for dv
    dq, dk, dv_ = _run(q, k, v, do, off, causal, base, "split_half")
    rq, rk, rv = OA.attention_backward(q, k, v, do, causal=causal, rope_base=base,
                                       operand_dtype=dtype, q_offset=off)
    assert float(abs(rq).max()) < 1e-12 and float(abs(rk).max()) < 1e-12
    atol = 1e-5 if dtype == "f32" else 2e-2
    assert float(dq.abs().max()) <= atol and float(dk.abs().max()) <= atol
    assert_grad_close(to_np(dv_), rv, f"edge {dtype} dv", **({} if dtype == "bf16" else F32_TOL))


FP32_CASES = [
    # (B, Hq, Hkv, Tq, Tk, q_offset, d, dv, causal, rope_base, layout)
    (2, 4, 1, 16, 64, 48, 16, 16, True, 10000.0, "split_half"),
    (1, 2, 2, 33, 70, 37, 32, 32, True, 10000.0, "adjacent"),
    (1, 6, 2, 20, 45, 0, 64, 64, False, 0.0, "split_half"),
    (1, 4, 4, 1, 300, 299, 128, 128, True, 10000.0, "split_half"),
    (1, 4, 2, 50, 40, 30, 64, 64, True, 10000.0, "split_half"),   # rows past the last key
    (1, 2, 1, 20, 90, 10, 32, 32, True, 10000.0, "split_half"),   # keys no query sees
    (2, 4, 1, 16, 64, 48, 16, 128, True, 10000.0, "split_half"),  # TPR from dv, 2 q channels
    (1, 2, 2, 33, 70, 37, 128, 16, True, 10000.0, "adjacent"),    # 2 v channels
    (1, 6, 2, 40, 45, 0, 32, 64, False, 0.0, "split_half"),
    (1, 4, 1, 70, 9, 5, 64, 32, False, 10000.0, "split_half"),
]


@pytest.mark.parametrize("B,hq,hkv,Tq,Tk,off,d,dv,causal,base,layout", FP32_CASES)
def test_bwd_ext_fp32(B, hq, hkv, Tq, Tk, off, d, dv, causal, base, layout):
    q, k, v, do = _inputs(B, hq, hkv, Tq, Tk, d, dv, "f32", seed=Tq + 5 * Tk + off + d + 7 * dv)
    _check(q, k, v, do, off, causal, base, layout, "f32", "fp32")


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("bf16", 64), ("f32", 32)])
def test_bwd_ext_square_equals_bwd(dtype, d):
    """Tq = Tk = T, q_offset = 0 and dv = d is csattn_attn_bwd: the same kernels, the
    same results bit for bit."""
    B, hq, hkv, T, base = 2, 4, 2, 200, 10000.0
    q, k, v, do = (t.to(dev()) for t in _inputs(B, hq, hkv, T, T, d, d, dtype, seed=17 + d))
    lse = torch.empty(B, hq, T, dtype=torch.float32, device=dev())
    out = csattn.attn_fwd(q, k, v, rope_base=base, lse=lse)
    a = csattn.attn_bwd(q, k, v, out, do, lse, rope_base=base)
    b = csattn.attn_bwd_ext(q, k, v, out, do, lse, rope_base=base)
    csattn.check_status()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_bwd_ext_chunk_rows_match_full_sequence():
    """The gradient of a chunk's loss is the full sequence's gradient restricted to
    that loss: with dout zero outside rows q_offset.., the full-sequence backward's dq
    rows q_offset.. and its dk, dv equal the chunk call's (both checked against the
    oracle, and against each other to the bf16 bound)."""
    B, hq, hkv, T, off, d = 1, 4, 2, 384, 200, 128
    q, k, v, do = _inputs(B, hq, hkv, T, T, d, d, "bf16", seed=5)
    do[:, :, :off] = 0
    full = _run(q, k, v, do, 0, True, 10000.0, "split_half")
    chunk = _run(q[:, :, off:].contiguous(), k, v, do[:, :, off:].contiguous(), off, True,
                 10000.0, "split_half")
    assert_grad_close(to_np(chunk[0]), to_np(full[0][:, :, off:]), "dq chunk vs full")
    assert_grad_close(to_np(chunk[1]), to_np(full[1]), "dk chunk vs full")
    assert_grad_close(to_np(chunk[2]), to_np(full[2]), "dv chunk vs full")
    rq, rk, rv = OA.attention_backward(q[:, :, off:], k, v, do[:, :, off:], causal=True,
                                       rope_base=10000.0, operand_dtype="bf16", q_offset=off)
    assert_grad_close(to_np(chunk[0]), rq, "dq chunk")
    assert_grad_close(to_np(chunk[1]), rk, "dk chunk")
    assert_grad_close(to_np(chunk[2]), rv, "dv chunk")


def test_bwd_ext_llama_chunk_workload_one_group():
    """The bench's chunk workload at full size (B=4, Hq=32, Hkv=8, 1024 queries at offset
    3072, Tk=4096, d=128, RoPE 1e4): one KV group (4 query heads) of one sequence against
    the oracle."""
    import attn_workloads as W
    wc = W.WORKLOADS["llama_chunk_bf16"]
    q, k, v = W.make_chunk_inputs(wc)
    g = torch.Generator()
    g.manual_seed(31)
    do = torch.randn(q.shape, generator=g).to(torch.bfloat16)
    dq, dk, dv = _run(q, k, v, do, wc.q_offset, True, wc.rope_base, "split_half")
    b, grp = 3, 6
    rep = wc.Hq // wc.Hkv
    hs = slice(grp * rep, (grp + 1) * rep)
    rq, rk, rv = OA.attention_backward(q[b:b + 1, hs], k[b:b + 1, grp:grp + 1],
                                       v[b:b + 1, grp:grp + 1], do[b:b + 1, hs], causal=True,
                                       rope_base=wc.rope_base, scale=wc.scale,
                                       operand_dtype="bf16", q_offset=wc.q_offset)
    assert_grad_close(to_np(dq[b:b + 1, hs]), rq, "dq chunk group")
    assert_grad_close(to_np(dk[b:b + 1, grp:grp + 1]), rk, "dk chunk group")
    assert_grad_close(to_np(dv[b:b + 1, grp:grp + 1]), rv, "dv chunk group")
