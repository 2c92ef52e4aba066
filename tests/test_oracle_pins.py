"""Pins of the CPU oracle against what the pages and the mathematics fix (no GPU).

Each ``pin_*`` function checks one fact through the public functions of
``oracle.attn``; the ``test_planted_*`` tests replace one oracle step by a
plausible mistake (on the CPU, in the oracle) and show that some pin fails.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import attn_workloads as W
from oracle import attn as OA
from oracle import naive as ON

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _facts():
    with open(os.path.join(GOLDEN, "page_facts.json")) as f:
        return json.load(f)


def _rand(shape, seed, mult=1.0):
    g = np.random.default_rng(seed)
    return g.standard_normal(shape) * mult


def _to_list(x):
    return np.asarray(x, dtype=np.float64).tolist()


# --------------------------------------------------------------------------- pins

def pin_softmax_page_example(o):
    f = _facts()["softmax_example"]
    p = o.softmax_rows(np.array([f["input"]]))[0]
    assert np.allclose(p, f["printed"], atol=0.5 * 10 ** (-f["printed_decimals"]))
    e = math.e
    exact = [e * e / (e * e + e + 1), e / (e * e + e + 1), 1 / (e * e + e + 1)]
    assert np.allclose(p, exact, rtol=0, atol=1e-15)


def pin_rows_sum_to_one(o):
    q = _rand((1, 3, 37, 8), 1)
    k = _rand((1, 3, 37, 8), 2)
    s = o.attention_scores(q[0], k[0], 0.3) + o.causal_additive_mask(37, 37)
    p = o.softmax_rows(s)
    assert np.all(np.abs(p.sum(-1) - 1.0) < 1e-12)
    assert np.all(p >= 0)


def pin_masked_weight_exactly_zero(o):
    q = _rand((23, 8), 3)
    k = _rand((23, 8), 4)
    s = o.attention_scores(q, k, 0.5) + o.causal_additive_mask(23, 23)
    p = o.softmax_rows(s)
    iu = np.triu_indices(23, 1)
    assert np.all(p[iu] == 0.0)
    assert np.all(p[np.tril_indices(23)] > 0.0)


def pin_mask_variants_differ(o):
    q = _rand((1, 1, 12, 8), 5)
    k = _rand((1, 1, 12, 8), 6)
    v = _rand((1, 1, 12, 8), 7)
    ref = o.attention(q, k, v, causal=True)
    s = o.attention_scores(q[0, 0], k[0, 0], 1 / math.sqrt(8))
    zero_mask = o.softmax_rows(s + np.where(np.triu(np.ones((12, 12)), 1) > 0, 0.0, 0.0)) @ v[0, 0]
    p_full = o.softmax_rows(s)
    p_after = np.where(np.triu(np.ones((12, 12)), 1) > 0, 0.0, p_full)
    after = p_after @ v[0, 0]
    assert np.max(np.abs(zero_mask - ref[0, 0])) > 1e-3
    assert np.max(np.abs(after - ref[0, 0])) > 1e-3
    assert np.all(p_after.sum(-1)[:-1] < 1.0 - 1e-6)


def pin_gqa_equals_mha_repeated(o):
    for rep in (1, 2, 4):
        Hkv = 2
        q = _rand((2, Hkv * rep, 19, 16), 10 + rep)
        k = _rand((2, Hkv, 19, 16), 20 + rep)
        v = _rand((2, Hkv, 19, 16), 30 + rep)
        a = o.attention(q, k, v, causal=True, rope_base=10000.0)
        kr = np.repeat(k, rep, axis=1)
        vr = np.repeat(v, rep, axis=1)
        b = o.attention(q, kr, vr, causal=True, rope_base=10000.0)
        assert np.array_equal(a, b)
        # and head h of the grouped result equals a single-head run on KV head h // rep
        for h in range(Hkv * rep):
            c = o.attention(q[:, h:h + 1], k[:, h // rep:h // rep + 1], v[:, h // rep:h // rep + 1],
                            causal=True, rope_base=10000.0)
            assert np.array_equal(a[:, h:h + 1], c)


def pin_basis_invariance(o):
    q = _rand((17, 8), 40)
    k = _rand((21, 8), 41)
    rng = np.random.default_rng(42)
    while True:
        R = rng.standard_normal((8, 8))
        if np.linalg.cond(R) < 10:
            break
    s0 = o.attention_scores(q, k, 0.25)
    s1 = o.attention_scores(q @ R, k @ np.linalg.inv(R).T, 0.25)
    assert np.max(np.abs(s1 - s0)) <= 1e-10 * max(1.0, np.max(np.abs(s0)))


def pin_qq_symmetric(o):
    q = _rand((15, 8), 43)
    s = o.attention_scores(q, q, 1.0)
    assert np.array_equal(s, s.T)


def pin_rope_relative(o):
    d = 16
    qv = _rand((1, d), 50)
    kv = _rand((1, d), 51)
    for layout in ("split_half", "adjacent"):
        def score(m, n):
            qm = o.rope_rotate(qv, [m], 10000.0, layout)
            kn = o.rope_rotate(kv, [n], 10000.0, layout)
            return float(o.attention_scores(qm, kn, 1.0)[0, 0])
        a, b, c = score(5, 2), score(20, 17), score(20, 10)
        assert abs(a - b) < 1e-12
        assert abs(a - c) > 1e-3


def pin_rope_orthogonal(o):
    x = _rand((9, 32), 52)
    pos = np.arange(9) * 37
    for layout in ("split_half", "adjacent"):
        y = o.rope_rotate(x, pos, 500000.0, layout)
        assert np.allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-14)
        y0 = o.rope_rotate(x[:1], [0], 10000.0, layout)
        assert np.array_equal(y0, x[:1])


def pin_rope_layouts_permute(o):
    d = 16
    x = _rand((7, d), 53)
    perm = np.empty(d, dtype=int)  # adjacent position of each split-half channel
    perm[: d // 2] = np.arange(0, d, 2)
    perm[d // 2:] = np.arange(1, d, 2)
    xa = np.empty_like(x)
    xa[:, perm] = x
    ys = o.rope_rotate(x, np.arange(7) * 3, 10000.0, "split_half")
    ya = o.rope_rotate(xa, np.arange(7) * 3, 10000.0, "adjacent")
    assert np.allclose(ya[:, perm], ys, rtol=0, atol=1e-14)


def pin_rope_angle_formula(o):
    # theta_i = base^(-2i/d): pair 0 turns by exactly pos radians, pair i by pos*base^(-2i/d)
    d = 8
    x = np.zeros((1, d))
    x[0, 0] = 1.0
    y = o.rope_rotate(x, [3], 10000.0, "split_half")
    assert abs(y[0, 0] - math.cos(3.0)) < 1e-15 and abs(y[0, d // 2] - math.sin(3.0)) < 1e-15
    x = np.zeros((1, d))
    x[0, 2] = 1.0
    y = o.rope_rotate(x, [7], 10000.0, "split_half")
    ang = 7 * 10000.0 ** (-4.0 / d)
    assert abs(y[0, 2] - math.cos(ang)) < 1e-15 and abs(y[0, 2 + d // 2] - math.sin(ang)) < 1e-15


def pin_naive_agreement(o):
    cases = [
        dict(B=1, Hkv=2, rep=1, T=9, d=4, causal=True, base=10000.0, layout="split_half"),
        dict(B=2, Hkv=1, rep=2, T=7, d=16, causal=True, base=10000.0, layout="adjacent"),
        dict(B=1, Hkv=2, rep=4, T=16, d=4, causal=False, base=0.0, layout="split_half"),
        dict(B=1, Hkv=1, rep=4, T=11, d=16, causal=True, base=500000.0, layout="split_half"),
        dict(B=1, Hkv=2, rep=2, T=13, d=4, causal=False, base=10000.0, layout="adjacent"),
    ]
    for i, c in enumerate(cases):
        Hq = c["Hkv"] * c["rep"]
        q = _rand((c["B"], Hq, c["T"], c["d"]), 60 + i, 2.0)
        k = _rand((c["B"], c["Hkv"], c["T"], c["d"]), 70 + i, 2.0)
        v = _rand((c["B"], c["Hkv"], c["T"], c["d"]), 80 + i)
        for rnd in (False, True):
            a = o.attention(q, k, v, causal=c["causal"], rope_base=c["base"], scale=0.37,
                            rope_layout=c["layout"], operand_dtype="bf16" if rnd else None)
            b = np.array(ON.naive_attention(_to_list(q), _to_list(k), _to_list(v), c["causal"],
                                            c["base"], 0.37, c["layout"], round_bf16=rnd))
            assert np.max(np.abs(a - b)) < 1e-12, (i, rnd, np.max(np.abs(a - b)))


def pin_value_width(o):
    """Values of another width than the keys ("Scaled dot-product attention": the weights
    come from q and k alone): agreement with the scalar loops for d_v != d_k, default
    scale 1/sqrt(d_k), and a single visible key returns its value row exactly."""
    for i, (dk, dv, causal, base) in enumerate([(4, 16, True, 10000.0), (16, 4, False, 0.0),
                                               (8, 2, True, 500000.0)]):
        q = _rand((1, 4, 7, dk), 300 + i, 2.0)
        k = _rand((1, 2, 9, dk), 310 + i, 2.0)
        v = _rand((1, 2, 9, dv), 320 + i)
        a = o.attention(q, k, v, causal=causal, rope_base=base, q_offset=2)
        b = np.array(ON.naive_attention(_to_list(q), _to_list(k), _to_list(v), causal, base, None,
                                        "split_half", q_offset=2))
        assert a.shape == (1, 4, 7, dv)
        assert np.max(np.abs(a - b)) < 1e-12, (i, np.max(np.abs(a - b)))
    q = _rand((1, 2, 1, 8), 330)
    k = _rand((1, 2, 1, 8), 331)
    v = _rand((1, 2, 1, 24), 332)
    assert np.array_equal(o.attention(q, k, v, causal=False), v)


def pin_cache_append_positions(o):
    """Appending a sequence to an empty cache in chunks puts at row t the key rotated at
    position t (the whole sequence rotated at once) and the value itself."""
    B, Hkv, d, Lmax = 2, 2, 8, 20
    k = _rand((B, Hkv, 16, d), 340)
    v = _rand((B, Hkv, 16, d), 341)
    kc = np.full((B, Hkv, Lmax, d), np.nan)
    vc = np.full((B, Hkv, Lmax, d), np.nan)
    L = 0
    for a, b in ((0, 5), (5, 12), (12, 16)):
        kc, vc = o.cache_append(k[:, :, a:b], v[:, :, a:b], kc, vc, [L, L], rope_base=10000.0,
                                operand_dtype="bf16")
        L = b
    want = o.round_to_bf16(o.rope_rotate(k, np.arange(16), 10000.0))
    assert np.array_equal(kc[:, :, :16], want)
    assert np.array_equal(vc[:, :, :16], v)
    assert np.all(np.isnan(kc[:, :, 16:])) and np.all(np.isnan(vc[:, :, 16:]))


def pin_cache_append_matches_decode_step(o):
    """One appended token writes the same cache rows as the decode step's append."""
    B, Hq, Hkv, d, Lmax = 3, 4, 2, 8, 12
    kc = _rand((B, Hkv, Lmax, d), 350)
    vc = _rand((B, Hkv, Lmax, d), 351)
    q1 = _rand((B, Hq, 1, d), 352)
    k1 = _rand((B, Hkv, 1, d), 353)
    v1 = _rand((B, Hkv, 1, d), 354)
    lens = [0, 5, 11]
    _, kd, vd = o.decode_step(q1, k1, v1, kc, vc, lens, rope_base=10000.0,
                              rope_layout="adjacent", operand_dtype="bf16")
    ka, va = o.cache_append(k1, v1, kc, vc, lens, rope_base=10000.0, rope_layout="adjacent",
                            operand_dtype="bf16")
    assert np.array_equal(ka, kd) and np.array_equal(va, vd)


def pin_cache_append_paged_equals_contiguous(o):
    """Appending into shuffled pages and gathering them back through the block table
    gives the contiguous append."""
    B, Hkv, d, page, n_lp = 2, 2, 8, 4, 4
    kc = np.zeros((B, Hkv, n_lp * page, d))
    vc = np.zeros((B, Hkv, n_lp * page, d))
    kn = _rand((B, Hkv, 6, d), 360)
    vn = _rand((B, Hkv, 6, d), 361)
    lens = [3, 9]
    perm = np.random.default_rng(362).permutation(B * n_lp + 1)
    table = perm[:B * n_lp].reshape(B, n_lp)
    kp = np.zeros((B * n_lp + 1, Hkv, page, d))
    vp = np.zeros((B * n_lp + 1, Hkv, page, d))
    kc2, vc2 = o.cache_append(kn, vn, kc, vc, lens, rope_base=10000.0)
    kp2, vp2 = o.cache_append_paged(kn, vn, kp, vp, table, lens, page, rope_base=10000.0)
    for b in range(B):
        for r in range(n_lp * page):
            assert np.array_equal(kp2[table[b, r // page], :, r % page], kc2[b, :, r])
            assert np.array_equal(vp2[table[b, r // page], :, r % page], vc2[b, :, r])


def pin_prefill_paged_equals_chunk(o):
    """A chunk over a paged cache of rotated keys (shuffled pages, NaN in every row
    past a sequence's end) equals the chunk of the contiguous definition: query i at
    position L_b + i over keys 0..L_b + i, per sequence, RoPE on both sides."""
    B, Hq, Hkv, d, Tq, page, n_lp = 3, 4, 2, 8, 4, 4, 5
    lens = [0, 5, 11]
    q = _rand((B, Hq, Tq, d), 370)
    k = _rand((B, Hkv, n_lp * page, d), 371)
    v = _rand((B, Hkv, n_lp * page, d), 372)
    kr = o.round_to_bf16(o.rope_rotate(k, np.arange(n_lp * page), 10000.0))
    perm = np.random.default_rng(373).permutation(B * n_lp + 2)
    table = perm[:B * n_lp].reshape(B, n_lp)
    kp = np.full((B * n_lp + 2, Hkv, page, d), np.nan)
    vp = np.full((B * n_lp + 2, Hkv, page, d), np.nan)
    for b, L in enumerate(lens):
        for t in range(L + Tq):
            kp[table[b, t // page], :, t % page] = kr[b, :, t]
            vp[table[b, t // page], :, t % page] = v[b, :, t]
    for causal in (True, False):
        got, got_lse = o.prefill_paged(q, kp, vp, table, lens, page, causal=causal,
                                       rope_base=10000.0, operand_dtype="bf16", lse=True)
        assert got.shape == (B, Hq, Tq, d)
        for b, L in enumerate(lens):
            sl = slice(0, L + Tq)
            want = o.attention(q[b:b + 1], k[b:b + 1, :, sl], v[b:b + 1, :, sl], causal=causal,
                               rope_base=10000.0, operand_dtype="bf16", q_offset=L)
            assert np.max(np.abs(got[b] - want[0])) < 1e-12, (causal, b)
            want_lse = o.attention_lse(q[b:b + 1], k[b:b + 1, :, sl], causal=causal,
                                       rope_base=10000.0, operand_dtype="bf16", q_offset=L)
            assert np.max(np.abs(got_lse[b] - want_lse[0])) < 1e-12, (causal, b)


def pin_degenerate_cases(o):
    q = _rand((1, 2, 1, 8), 90)
    k = _rand((1, 2, 1, 8), 91)
    v = _rand((1, 2, 1, 8), 92)
    assert np.array_equal(o.attention(q, k, v, causal=False), v)
    q = _rand((1, 2, 6, 8), 93)
    k = _rand((1, 2, 6, 8), 94)
    v = _rand((1, 2, 6, 8), 95)
    out = o.attention(q, k, v, causal=True, rope_base=10000.0)
    assert np.array_equal(out[:, :, 0], v[:, :, 0])


def pin_decode_equals_prefill_last_row(o):
    B, Hkv, rep, d = 3, 2, 2, 16
    T = 29
    q = _rand((B, Hkv * rep, T, d), 100)
    k = _rand((B, Hkv, T, d), 101)
    v = _rand((B, Hkv, T, d), 102)
    full = o.attention(q, k, v, causal=True, rope_base=10000.0)
    qr = o.rope_rotate(q, np.arange(T), 10000.0)
    kr = o.rope_rotate(k, np.arange(T), 10000.0)
    lens = [T, 17, 1]
    Lmax = T + 3
    kc = np.full((B, Hkv, Lmax, d), np.nan)
    vc = np.full((B, Hkv, Lmax, d), np.nan)
    qd = np.empty((B, Hkv * rep, 1, d))
    for b, L in enumerate(lens):
        kc[b, :, :L] = kr[b, :, :L]
        vc[b, :, :L] = v[b, :, :L]
        qd[b, :, 0] = qr[b, :, L - 1]
    dec = o.decode(qd, kc, vc, lens)
    assert not np.any(np.isnan(dec))
    for b, L in enumerate(lens):
        ref = o.attention(q[b:b + 1, :, :L], k[b:b + 1, :, :L], v[b:b + 1, :, :L],
                          causal=True, rope_base=10000.0)
        assert np.max(np.abs(dec[b, :, 0] - ref[0, :, L - 1])) < 1e-12
    assert np.max(np.abs(dec[0, :, 0] - full[0, :, T - 1])) < 1e-12
    nd = np.array(ON.naive_decode(_to_list(qd[:, :, 0]), np.nan_to_num(kc).tolist(),
                                  np.nan_to_num(vc).tolist(), lens))
    assert np.max(np.abs(nd - dec[:, :, 0])) < 1e-12


def pin_merge_partials(o):
    s = _rand((97,), 110, 3.0)
    v = _rand((97, 8), 111)
    ref = o.softmax_rows(s[None])[0] @ v
    for bounds in ([0, 97], [0, 10, 97], [0, 32, 64, 96, 97], [0, 0, 50, 97, 97], [0, 1, 2, 97]):
        ms, ls, os_ = o.split_partials(s, v, bounds)
        out = o.merge_partials(ms, ls, os_)
        assert np.max(np.abs(out - ref)) < 1e-12


def pin_bf16_rounding(o):
    g = torch.Generator().manual_seed(5)
    x32 = torch.randn(20000, generator=g) * torch.exp2(torch.randint(-20, 20, (20000,), generator=g).float())
    x32 = torch.cat([x32, torch.tensor([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 0.0, 2 ** -130,
                                        3.0e38, 65504.0])])
    ref = x32.to(torch.bfloat16).double().numpy()
    got = o.round_to_bf16(x32.double().numpy())
    assert np.array_equal(got, ref)
    x64 = _rand((300,), 120, 10.0)
    naive = np.array([ON.naive_round_bf16(float(t)) for t in x64])
    assert np.array_equal(o.round_to_bf16(x64), naive)


def pin_chunk_equals_full_rows(o):
    """A chunk of queries after a cache prefix (q_offset) gives the same rows as the
    full causal prefill ("The Transformer architecture", "Hands-on": the query at
    position p sees keys 0..p, rotated at p)."""
    B, Hkv, rep, T, d = 1, 2, 2, 40, 16
    q = _rand((B, Hkv * rep, T, d), 130, 2.0)
    k = _rand((B, Hkv, T, d), 131, 2.0)
    v = _rand((B, Hkv, T, d), 132)
    for dt in (None, "bf16"):
        full = o.attention(q, k, v, causal=True, rope_base=10000.0, operand_dtype=dt)
        for off in (0, 7, 23, 39):
            chunk = o.attention(q[:, :, off:], k, v, causal=True, rope_base=10000.0,
                                operand_dtype=dt, q_offset=off)
            assert chunk.shape == (B, Hkv * rep, T - off, d)
            assert np.max(np.abs(chunk - full[:, :, off:])) < 1e-12, (dt, off)
        # a chunk that stops early: keys past the chunk's last position are never visible
        mid = o.attention(q[:, :, 10:20], k, v, causal=True, rope_base=10000.0, operand_dtype=dt,
                          q_offset=10)
        assert np.max(np.abs(mid - full[:, :, 10:20])) < 1e-12


def pin_chunk_naive(o):
    """Query offset and rectangular shapes against the scalar-loop oracle."""
    cases = [dict(Tq=4, Tk=9, off=5, causal=True, base=10000.0, layout="split_half"),
             dict(Tq=3, Tk=12, off=2, causal=True, base=10000.0, layout="adjacent"),
             dict(Tq=5, Tk=11, off=0, causal=False, base=0.0, layout="split_half"),
             dict(Tq=7, Tk=3, off=4, causal=False, base=10000.0, layout="split_half")]
    for i, c in enumerate(cases):
        q = _rand((1, 4, c["Tq"], 8), 140 + i, 2.0)
        k = _rand((1, 2, c["Tk"], 8), 150 + i, 2.0)
        v = _rand((1, 2, c["Tk"], 8), 160 + i)
        for rnd in (False, True):
            a = o.attention(q, k, v, causal=c["causal"], rope_base=c["base"], scale=0.41,
                            rope_layout=c["layout"], operand_dtype="bf16" if rnd else None,
                            q_offset=c["off"])
            b = np.array(ON.naive_attention(_to_list(q), _to_list(k), _to_list(v), c["causal"],
                                            c["base"], 0.41, c["layout"], round_bf16=rnd,
                                            q_offset=c["off"]))
            assert np.max(np.abs(a - b)) < 1e-12, (i, rnd)
            rows = np.arange(c["Tq"])[::2]
            r = o.attention_rows(q, k, v, 0, 3, rows, causal=c["causal"], rope_base=c["base"],
                                 scale=0.41, rope_layout=c["layout"],
                                 operand_dtype="bf16" if rnd else None, q_offset=c["off"])
            assert np.max(np.abs(r - a[0, 3, rows])) < 1e-12
    # one key: every query returns that key's value exactly
    q = _rand((1, 2, 6, 8), 170)
    k = _rand((1, 1, 1, 8), 171)
    v = _rand((1, 1, 1, 8), 172)
    out = o.attention(q, k, v, causal=False, rope_base=10000.0, q_offset=3)
    assert np.array_equal(out, np.broadcast_to(v, (1, 2, 6, 8)))


def pin_decode_is_chunk_of_one(o):
    """Decode at length L equals a one-query chunk at q_offset = L - 1."""
    B, Hkv, rep, d, L = 1, 2, 4, 16, 23
    q = _rand((B, Hkv * rep, L, d), 180)
    k = _rand((B, Hkv, L, d), 181)
    v = _rand((B, Hkv, L, d), 182)
    one = o.attention(q[:, :, L - 1:], k, v, causal=True, rope_base=10000.0, q_offset=L - 1)
    qd = o.rope_rotate(q[:, :, L - 1:], np.array([L - 1]), 10000.0)
    kr = o.rope_rotate(k, np.arange(L), 10000.0)
    dec = o.decode(qd, kr, v, [L])
    assert np.max(np.abs(one - dec)) < 1e-12


def pin_decode_step_appends_then_attends(o):
    """Appending the new token's rotated key and value at row cache_len and attending
    over rows 0..cache_len equals a one-query chunk over the whole unrotated sequence."""
    B, Hkv, rep, d, Lmax = 3, 2, 2, 16, 40
    lens = [0, 17, 38]
    for dt in (None, "bf16"):
        kc = np.full((B, Hkv, Lmax, d), np.nan)
        vc = np.full((B, Hkv, Lmax, d), np.nan)
        seqs = []
        for b, L in enumerate(lens):
            K = _rand((1, Hkv, L + 1, d), 190 + b, 2.0)
            V = _rand((1, Hkv, L + 1, d), 195 + b)
            Q = _rand((1, Hkv * rep, 1, d), 200 + b, 2.0)
            kc[b, :, :L] = o.round_to(o.rope_rotate(K[0, :, :L], np.arange(L), 10000.0), dt)
            vc[b, :, :L] = V[0, :, :L]
            seqs.append((K, V, Q))
        qn = np.concatenate([s_[2] for s_ in seqs])
        kn = np.concatenate([s_[0][:, :, -1:] for s_ in seqs])
        vn = np.concatenate([s_[1][:, :, -1:] for s_ in seqs])
        out, kc2, vc2 = o.decode_step(qn, kn, vn, kc, vc, lens, rope_base=10000.0,
                                      operand_dtype=dt)
        for b, L in enumerate(lens):
            K, V, Q = seqs[b]
            ref = o.attention(Q, K, V, causal=True, rope_base=10000.0, operand_dtype=dt,
                              q_offset=L)
            assert np.max(np.abs(out[b] - ref[0])) < 1e-12, (dt, b)
            assert np.array_equal(vc2[b, :, L], V[0, :, L])
            rk = o.round_to(o.rope_rotate(K[0, :, L:L + 1], np.array([L]), 10000.0), dt)
            assert np.array_equal(kc2[b, :, L], rk[:, 0])
            assert np.all(np.isnan(kc2[b, :, L + 1:])) and np.all(np.isnan(vc2[b, :, L + 1:]))
            assert np.array_equal(kc2[b, :, :L], kc[b, :, :L])


def _fd_grads(o, q, k, v, do, kw, h=1e-6):
    """Central finite differences of sum(attention(q, k, v) * do) in float64."""
    def f(a, b, c):
        return float(np.sum(o.attention(a, b, c, **kw) * do))
    grads = []
    for which in range(3):
        args = [q, k, v]
        x = args[which]
        gx = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            ap, am = list(args), list(args)
            ap[which], am[which] = xp, xm
            gx[idx] = (f(*ap) - f(*am)) / (2 * h)
        grads.append(gx)
    return grads


def pin_backward_finite_differences(o):
    """The gradients of the backward agree with central differences of the forward."""
    cases = [dict(Hq=4, Hkv=2, T=7, d=8, kw=dict(causal=True, rope_base=100.0, scale=0.4)),
             dict(Hq=2, Hkv=1, T=6, d=4, kw=dict(causal=False, rope_base=50.0, scale=0.7,
                                                 rope_layout="adjacent")),
             dict(Hq=2, Hkv=2, T=5, d=4, kw=dict(causal=True, rope_base=0.0, scale=0.5))]
    for i, c in enumerate(cases):
        q = _rand((1, c["Hq"], c["T"], c["d"]), 210 + i)
        k = _rand((1, c["Hkv"], c["T"], c["d"]), 220 + i)
        v = _rand((1, c["Hkv"], c["T"], c["d"]), 230 + i)
        do = _rand((1, c["Hq"], c["T"], c["d"]), 240 + i)
        got = o.attention_backward(q, k, v, do, **c["kw"])
        num = _fd_grads(o, q, k, v, do, c["kw"])
        for name, a, b in zip("qkv", got, num):
            assert np.max(np.abs(a - b)) < 1e-7, (i, name, np.max(np.abs(a - b)))
    # a chunk at an offset: the query rotation and the mask both move
    q = _rand((1, 2, 4, 8), 250)
    k = _rand((1, 1, 9, 8), 251)
    v = _rand((1, 1, 9, 8), 252)
    do = _rand((1, 2, 4, 8), 253)
    kw = dict(causal=True, rope_base=100.0, scale=0.45, q_offset=5)
    got = o.attention_backward(q, k, v, do, **kw)
    for name, a, b in zip("qkv", got, _fd_grads(o, q, k, v, do, kw)):
        assert np.max(np.abs(a - b)) < 1e-7, ("offset", name)
    # values of their own width: a chunk (d_v > d_k) and an unmasked rectangle (d_v < d_k,
    # Tq > Tk) with RoPE at an offset
    for tag, shp, kw in (("dv>dk", (2, 1, 3, 7, 4, 6), dict(causal=True, rope_base=100.0,
                                                            scale=0.5, q_offset=4)),
                         ("rect", (2, 2, 5, 3, 8, 4), dict(causal=False, rope_base=60.0,
                                                           scale=0.35, q_offset=2,
                                                           rope_layout="adjacent"))):
        hq, hkv, tq, tk, dk, dv = shp
        q = _rand((1, hq, tq, dk), 254)
        k = _rand((1, hkv, tk, dk), 255)
        v = _rand((1, hkv, tk, dv), 256)
        do = _rand((1, hq, tq, dv), 257)
        got = o.attention_backward(q, k, v, do, **kw)
        assert got[0].shape == q.shape and got[1].shape == k.shape and got[2].shape == v.shape
        for name, a, b in zip("qkv", got, _fd_grads(o, q, k, v, do, kw)):
            assert np.max(np.abs(a - b)) < 1e-7, (tag, name, np.max(np.abs(a - b)))


def pin_backward_autograd(o):
    """Against torch autograd (float64) of a forward written here with plain torch ops."""
    B, Hq, Hkv, T, d, base, sc = 2, 6, 2, 33, 16, 10000.0, 0.3
    q = torch.tensor(_rand((B, Hq, T, d), 260), requires_grad=True)
    k = torch.tensor(_rand((B, Hkv, T, d), 261), requires_grad=True)
    v = torch.tensor(_rand((B, Hkv, T, d), 262), requires_grad=True)
    do = torch.tensor(_rand((B, Hq, T, d), 263))
    pos = torch.arange(T, dtype=torch.float64)
    ang = pos[:, None] * base ** (-torch.arange(0, d, 2, dtype=torch.float64) / d)[None, :]
    cos, sin = torch.cos(ang), torch.sin(ang)

    def rot(x):
        a, b = x[..., : d // 2], x[..., d // 2:]
        return torch.cat([a * cos - b * sin, a * sin + b * cos], dim=-1)

    kf = rot(k).repeat_interleave(Hq // Hkv, dim=1)
    vf = v.repeat_interleave(Hq // Hkv, dim=1)
    s_ = rot(q) @ kf.transpose(-1, -2) * sc
    s_ = s_.masked_fill(torch.triu(torch.ones(T, T, dtype=torch.bool), 1), float("-inf"))
    out = torch.softmax(s_, dim=-1) @ vf
    (out * do).sum().backward()
    got = o.attention_backward(q.detach().numpy(), k.detach().numpy(), v.detach().numpy(),
                               do.numpy(), causal=True, rope_base=base, scale=sc)
    for a, t in zip(got, (q.grad, k.grad, v.grad)):
        assert np.max(np.abs(a - t.numpy())) < 1e-12


def pin_rope_transpose_inverts(o):
    x = _rand((3, 11, 16), 270)
    y = _rand((3, 11, 16), 271)
    pos = np.arange(11) * 37
    for layout in ("split_half", "adjacent"):
        r = o.rope_rotate(x, pos, 10000.0, layout)
        assert np.max(np.abs(o.rope_rotate_transpose(r, pos, 10000.0, layout) - x)) < 1e-13
        # <R x, y> = <x, R^T y>
        lhs = np.sum(r * y)
        rhs = np.sum(x * o.rope_rotate_transpose(y, pos, 10000.0, layout))
        assert abs(lhs - rhs) < 1e-10


def pin_decode_paged_equals_contiguous(o):
    """A contiguous cache scattered into shuffled pages decodes to the same result."""
    B, Hkv, rep, d, page = 3, 2, 2, 8, 4
    lens = [1, 9, 12]
    n_lp = 3  # logical pages per sequence
    kc = _rand((B, Hkv, n_lp * page, d), 280)
    vc = _rand((B, Hkv, n_lp * page, d), 281)
    q = _rand((B, Hkv * rep, 1, d), 282)
    perm = np.random.default_rng(283).permutation(B * n_lp + 2)  # two spare pages
    kp = np.full((B * n_lp + 2, Hkv, page, d), np.nan)
    vp = np.full((B * n_lp + 2, Hkv, page, d), np.nan)
    table = np.zeros((B, n_lp), dtype=np.int32)
    for b in range(B):
        for lp in range(n_lp):
            pp = perm[b * n_lp + lp]
            table[b, lp] = pp
            kp[pp] = kc[b, :, lp * page:(lp + 1) * page]
            vp[pp] = vc[b, :, lp * page:(lp + 1) * page]
    got = o.decode_paged(q, kp, vp, table, lens, page)
    assert np.max(np.abs(got - o.decode(q, kc, vc, lens))) < 1e-12


def pin_lse_normalises_softmax(o):
    """The log-sum-exp is the log of the softmax denominator ("The Transformer
    architecture", "Softmax is a differentiable allocation"): exp(S*scale + M - lse)
    is the softmax row itself and sums to 1 (GQA, RoPE, a query offset, causal and not).
    S is formed here from the rotated operands with a plain matrix product."""
    B, Hq, Hkv, Tq, Tk, d, sc, off = 2, 4, 2, 9, 14, 8, 0.41, 5
    q = _rand((B, Hq, Tq, d), 400, 2.0)
    k = _rand((B, Hkv, Tk, d), 401, 2.0)
    qr = o.rope_rotate(q, off + np.arange(Tq), 10000.0)
    kr = o.rope_rotate(k, np.arange(Tk), 10000.0)
    for causal in (True, False):
        lse = o.attention_lse(q, k, causal=causal, rope_base=10000.0, scale=sc, q_offset=off)
        assert lse.shape == (B, Hq, Tq)
        for b in range(B):
            for h in range(Hq):
                s = (qr[b, h] @ kr[b, h // (Hq // Hkv)].T) * sc
                if causal:
                    s = np.where(np.arange(Tk)[None, :] > off + np.arange(Tq)[:, None], -np.inf, s)
                p = np.exp(s - lse[b, h][:, None])
                assert np.all(np.abs(p.sum(-1) - 1.0) < 1e-12), (causal, b, h)
                assert np.max(np.abs(p - o.softmax_rows(s))) < 1e-12


def pin_lse_closed_forms(o):
    """One visible key: lse = its score.  Two visible keys with equal scores s:
    lse = s + ln 2.  Causal row 0 sees key 0 only; with k[1] = k[0] and no RoPE,
    row 1 sees two equal scores."""
    q = _rand((1, 2, 4, 8), 410)
    k = _rand((1, 1, 4, 8), 411)
    k[:, :, 1] = k[:, :, 0]
    sc = 0.3
    lse = o.attention_lse(q, k, causal=True, scale=sc)
    for h in range(2):
        s0 = float(q[0, h, 0] @ k[0, 0, 0]) * sc
        s1 = float(q[0, h, 1] @ k[0, 0, 0]) * sc
        assert abs(lse[0, h, 0] - s0) < 1e-13
        assert abs(lse[0, h, 1] - (s1 + math.log(2.0))) < 1e-13
    # decode-like chunk: one query at offset L-1 over L keys equals the last full row
    full = o.attention_lse(q, k, causal=True, scale=sc)
    last = o.attention_lse(q[:, :, 3:], k, causal=True, scale=sc, q_offset=3)
    assert np.max(np.abs(full[:, :, 3:] - last)) < 1e-13


def pin_lse_naive_agreement(o):
    """Against the scalar loops of ``oracle.naive.naive_lse`` (separately written), on the
    case grid of the output's brute-force pin plus a query offset and a rectangular case."""
    cases = [
        dict(B=1, Hkv=2, rep=1, T=9, Tk=9, d=4, causal=True, base=10000.0, layout="split_half", off=0),
        dict(B=2, Hkv=1, rep=2, T=7, Tk=7, d=16, causal=True, base=10000.0, layout="adjacent", off=0),
        dict(B=1, Hkv=2, rep=4, T=16, Tk=16, d=4, causal=False, base=0.0, layout="split_half", off=0),
        dict(B=1, Hkv=1, rep=4, T=11, Tk=11, d=16, causal=True, base=500000.0, layout="split_half",
             off=0),
        dict(B=1, Hkv=2, rep=2, T=13, Tk=13, d=4, causal=False, base=10000.0, layout="adjacent", off=0),
        dict(B=1, Hkv=2, rep=2, T=5, Tk=12, d=8, causal=True, base=10000.0, layout="split_half", off=7),
        dict(B=2, Hkv=1, rep=3, T=4, Tk=10, d=4, causal=False, base=10000.0, layout="adjacent", off=3),
    ]
    for i, c in enumerate(cases):
        Hq = c["Hkv"] * c["rep"]
        q = _rand((c["B"], Hq, c["T"], c["d"]), 420 + i, 2.0)
        k = _rand((c["B"], c["Hkv"], c["Tk"], c["d"]), 430 + i, 2.0)
        for rnd in (False, True):
            a = o.attention_lse(q, k, causal=c["causal"], rope_base=c["base"], scale=0.37,
                                rope_layout=c["layout"], operand_dtype="bf16" if rnd else None,
                                q_offset=c["off"])
            b = np.array(ON.naive_lse(_to_list(q), _to_list(k), c["causal"], c["base"], 0.37,
                                      c["layout"], round_bf16=rnd, q_offset=c["off"]))
            assert np.max(np.abs(a - b)) < 1e-12, (i, rnd, np.max(np.abs(a - b)))


ALL_PINS = [pin_softmax_page_example, pin_rows_sum_to_one, pin_masked_weight_exactly_zero,
            pin_mask_variants_differ, pin_gqa_equals_mha_repeated, pin_basis_invariance,
            pin_qq_symmetric, pin_rope_relative, pin_rope_orthogonal, pin_rope_layouts_permute,
            pin_rope_angle_formula, pin_naive_agreement, pin_degenerate_cases,
            pin_decode_equals_prefill_last_row, pin_merge_partials, pin_bf16_rounding,
            pin_chunk_equals_full_rows, pin_chunk_naive, pin_decode_is_chunk_of_one,
            pin_decode_step_appends_then_attends, pin_backward_finite_differences,
            pin_backward_autograd, pin_rope_transpose_inverts,
            pin_decode_paged_equals_contiguous, pin_value_width, pin_cache_append_positions,
            pin_cache_append_matches_decode_step, pin_cache_append_paged_equals_contiguous,
            pin_prefill_paged_equals_chunk, pin_lse_normalises_softmax, pin_lse_closed_forms,
            pin_lse_naive_agreement]

LSE_PINS = [pin_lse_normalises_softmax, pin_lse_closed_forms, pin_lse_naive_agreement]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(OA)


def test_score_variance_of_generator():
    w = W.WORKLOADS["llama_gqa_bf16"].with_(B=1, Hq=4, Hkv=1, T=512)
    q, k, _ = W.make_prefill_inputs(w)
    qd = q.double().numpy()[0, 0]
    kd = k.double().numpy()[0, 0]
    s = qd @ kd.T
    assert abs(np.var(s) / 128.0 - 1.0) < 0.05


def test_oracle_golden_regression():
    """Values written by tests/golden/make_oracle_golden.py (calls oracle/ only)."""
    with open(os.path.join(GOLDEN, "oracle_tiny_f32.json")) as f:
        g = json.load(f)
    w = W.WORKLOADS["tiny_f32"]
    q, k, v = W.make_prefill_inputs(w)
    out = OA.attention(q, k, v, causal=True, rope_base=w.rope_base, scale=w.scale,
                       operand_dtype="f32")
    for (b, h, t, c), val in zip(g["index"], g["value"]):
        assert abs(out[b, h, t, c] - val) < 1e-12


# ----------------------------------------------------------------- planted mistakes

class _Mutant:
    """The oracle module with one function replaced."""

    def __init__(self, **repl):
        self.__dict__.update({n: getattr(OA, n) for n in OA.__all__})
        self.__dict__.update(repl)
        me = self

        def attention(q, k, v, *, causal=True, rope_base=0.0, scale=None,
                      rope_layout="split_half", operand_dtype=None, q_offset=0):
            q = np.asarray(q, np.float64)
            k = np.asarray(k, np.float64)
            v = np.asarray(v, np.float64)
            B, Hq, T, d = q.shape
            Tk = k.shape[2]
            dsc = v.shape[-1] if "scale_from_v" in repl else d
            sc = 1 / math.sqrt(dsc) if (scale is None or scale <= 0) else scale
            if rope_base > 0:
                q = me.round_to(me.rope_rotate(q, q_offset + np.arange(T), rope_base, rope_layout),
                                operand_dtype)
                k = me.round_to(me.rope_rotate(k, np.arange(Tk), rope_base, rope_layout),
                                operand_dtype)
                if "rope_on_v" in repl:
                    v = me.rope_rotate(v, np.arange(Tk), rope_base, rope_layout)
            kf, vf = me.expand_kv_heads(k, Hq), me.expand_kv_heads(v, Hq)
            mask = me.causal_additive_mask(T, Tk, q_offset) if causal else 0.0
            out = np.empty((B, Hq, T, v.shape[-1]))
            for b in range(B):
                for h in range(Hq):
                    out[b, h] = me.softmax_rows(me.attention_scores(q[b, h], kf[b, h], sc) + mask) @ vf[b, h]
            return out

        if "attention" not in repl:
            self.attention = attention


def _fails(mutant, pins):
    failed = []
    for p in pins:
        try:
            p(mutant)
        except AssertionError:
            failed.append(p.__name__)
    return failed


def test_mutant_harness_is_faithful():
    assert _fails(_Mutant(), [pin_naive_agreement, pin_gqa_equals_mha_repeated,
                              pin_degenerate_cases, pin_rows_sum_to_one]) == []


def test_planted_gqa_modulo_mapping():
    def bad_expand(kv, n_q_heads):
        kv = np.asarray(kv, np.float64)
        return np.tile(kv, (1,) * (kv.ndim - 3) + (n_q_heads // kv.shape[-3], 1, 1))  # h % Hkv
    assert _fails(_Mutant(expand_kv_heads=bad_expand), [pin_naive_agreement])


def test_planted_softmax_wrong_axis():
    def bad_softmax(z):
        z = np.asarray(z, np.float64)
        e = np.exp(z - np.max(z, axis=-2, keepdims=True))
        return e / e.sum(axis=-2, keepdims=True)
    assert _fails(_Mutant(softmax_rows=bad_softmax), [pin_rows_sum_to_one])


def test_planted_mask_transposed():
    def bad_mask(tq, tk, q_offset=0):
        i = np.arange(tq)[:, None]
        j = np.arange(tk)[None, :]
        return np.where(j < i, -np.inf, 0.0)
    assert _fails(_Mutant(causal_additive_mask=bad_mask),
                  [pin_masked_weight_exactly_zero, pin_naive_agreement])


def test_planted_rope_sign():
    def bad_rope(x, positions, base, layout="split_half"):
        x = np.asarray(x, np.float64)
        d = x.shape[-1]
        c, s = OA.rope_cos_sin(positions, d, base)
        out = np.empty_like(x)
        a, b = x[..., : d // 2], x[..., d // 2:]
        out[..., : d // 2] = a * c + b * s
        out[..., d // 2:] = a * s + b * c
        return out
    assert _fails(_Mutant(rope_rotate=bad_rope), [pin_rope_orthogonal, pin_rope_relative])


def test_planted_rope_on_v():
    assert _fails(_Mutant(rope_on_v=True), [pin_naive_agreement])


def test_planted_dropped_scale():
    def bad_scores(q, k, scale):
        return np.asarray(q, np.float64) @ np.swapaxes(np.asarray(k, np.float64), -1, -2)
    assert _fails(_Mutant(attention_scores=bad_scores), [pin_naive_agreement])


def test_planted_rope_frequency_off_by_one():
    def bad_freq(d, base):
        i = np.arange(d // 2, dtype=np.float64)
        return np.power(float(base), -(2.0 * (i + 1)) / float(d))

    def bad_cs(positions, d, base):
        ang = np.outer(np.asarray(positions, np.float64), bad_freq(d, base))
        return np.cos(ang), np.sin(ang)

    def bad_rope(x, positions, base, layout="split_half"):
        x = np.asarray(x, np.float64)
        d = x.shape[-1]
        c, s = bad_cs(positions, d, base)
        out = np.empty_like(x)
        if layout == "split_half":
            a, b = x[..., : d // 2], x[..., d // 2:]
            out[..., : d // 2] = a * c - b * s
            out[..., d // 2:] = a * s + b * c
        else:
            a, b = x[..., 0::2], x[..., 1::2]
            out[..., 0::2] = a * c - b * s
            out[..., 1::2] = a * s + b * c
        return out
    assert _fails(_Mutant(rope_rotate=bad_rope), [pin_rope_angle_formula, pin_naive_agreement])


def test_planted_bf16_truncation():
    def bad_round(x, dtype):
        x = np.asarray(x, np.float64)
        if dtype != "bf16":
            return x
        m, e = np.frexp(x)
        return np.ldexp(np.trunc(np.ldexp(m, 8)), e - 8)
    assert _fails(_Mutant(round_to=bad_round), [pin_naive_agreement])



def _chunk_attention(q, k, v, mask_offset, rope_offset, causal=True, rope_base=0.0, scale=None,
                     rope_layout="split_half", operand_dtype=None):
    """The oracle's chunk definition with the mask and the RoPE positions offset separately."""
    q, k, v = (np.asarray(t, np.float64) for t in (q, k, v))
    B, Hq, Tq, d = q.shape
    Tk = k.shape[2]
    sc = 1 / math.sqrt(d) if (scale is None or scale <= 0) else scale
    if rope_base > 0:
        q = OA.round_to(OA.rope_rotate(q, rope_offset + np.arange(Tq), rope_base, rope_layout),
                        operand_dtype)
        k = OA.round_to(OA.rope_rotate(k, np.arange(Tk), rope_base, rope_layout), operand_dtype)
    kf, vf = OA.expand_kv_heads(k, Hq), OA.expand_kv_heads(v, Hq)
    mask = OA.causal_additive_mask(Tq, Tk, mask_offset) if causal else 0.0
    out = np.empty((B, Hq, Tq, v.shape[-1]))
    for b in range(B):
        for h in range(Hq):
            out[b, h] = OA.softmax_rows(OA.attention_scores(q[b, h], kf[b, h], sc) + mask) @ vf[b, h]
    return out


def test_chunk_helper_is_faithful():
    def good(q, k, v, *, q_offset=0, **kw):
        return _chunk_attention(q, k, v, q_offset, q_offset, **kw)
    assert _fails(_Mutant(attention=good), [pin_chunk_equals_full_rows, pin_chunk_naive,
                                            pin_decode_is_chunk_of_one]) == []


def test_planted_offset_ignored_by_mask():
    def bad(q, k, v, *, q_offset=0, **kw):
        return _chunk_attention(q, k, v, 0, q_offset, **kw)
    assert _fails(_Mutant(attention=bad), [pin_chunk_equals_full_rows])


def test_planted_offset_ignored_by_rope():
    def bad(q, k, v, *, q_offset=0, **kw):
        return _chunk_attention(q, k, v, q_offset, 0, **kw)
    assert _fails(_Mutant(attention=bad), [pin_chunk_equals_full_rows, pin_decode_is_chunk_of_one])


def test_planted_decode_step_rotates_key_at_wrong_position():
    def bad(q_new, k_new, v_new, k_cache, v_cache, cache_lens, *, rope_base=0.0,
            rope_layout="split_half", scale=None, operand_dtype=None):
        # the new key rotated at position cache_len + 1 instead of cache_len
        kc = np.array(k_cache, dtype=np.float64)
        vc = np.array(v_cache, dtype=np.float64)
        qr = np.empty(np.shape(q_new))
        lens = [int(x) for x in cache_lens]
        for b, pos in enumerate(lens):
            qr[b] = OA.round_to(OA.rope_rotate(np.asarray(q_new[b], np.float64), np.array([pos]),
                                               rope_base, rope_layout), operand_dtype)
            kr = OA.rope_rotate(np.asarray(k_new[b], np.float64), np.array([pos + 1]), rope_base,
                                rope_layout)
            kc[b, :, pos] = OA.round_to(kr, operand_dtype)[:, 0]
            vc[b, :, pos] = np.asarray(v_new[b], np.float64)[:, 0]
        return OA.decode(qr, kc, vc, [L + 1 for L in lens], scale=scale), kc, vc
    assert _fails(_Mutant(decode_step=bad), [pin_decode_step_appends_then_attends])


def _backward_variant(drop_d=False, last_head_only=False, forward_rotation=False):
    """The oracle's backward with one planted mistake."""
    def bwd(q, k, v, dout, *, causal=True, rope_base=0.0, scale=None, rope_layout="split_half",
            operand_dtype=None, q_offset=0):
        q, k, v, do = (np.asarray(t, np.float64) for t in (q, k, v, dout))
        B, Hq, T, d = q.shape
        Hkv, Tk = k.shape[1], k.shape[2]
        rep = Hq // Hkv
        sc = 1 / math.sqrt(d) if (scale is None or scale <= 0) else scale
        qpos, kpos = q_offset + np.arange(T), np.arange(Tk)
        qr = OA.rope_rotate(q, qpos, rope_base, rope_layout) if rope_base > 0 else q
        kr = OA.rope_rotate(k, kpos, rope_base, rope_layout) if rope_base > 0 else k
        mask = OA.causal_additive_mask(T, Tk, q_offset) if causal else 0.0
        dqr, dkr, dv = np.zeros_like(qr), np.zeros_like(kr), np.zeros_like(v)
        for b in range(B):
            for h in range(Hq):
                g = h // rep
                p = OA.softmax_rows(OA.attention_scores(qr[b, h], kr[b, g], sc) + mask)
                o = p @ v[b, g]
                keep = (h % rep == rep - 1) or not last_head_only
                if keep:
                    dv[b, g] += p.T @ do[b, h]
                dp = do[b, h] @ v[b, g].T
                dsc = p * dp if drop_d else p * (dp - np.sum(do[b, h] * o, -1, keepdims=True))
                dqr[b, h] = sc * dsc @ kr[b, g]
                if keep:
                    dkr[b, g] += sc * dsc.T @ qr[b, h]
        back = OA.rope_rotate if forward_rotation else OA.rope_rotate_transpose
        if rope_base > 0:
            return back(dqr, qpos, rope_base, rope_layout), back(dkr, kpos, rope_base, rope_layout), dv
        return dqr, dkr, dv
    return bwd


def test_backward_variant_helper_is_faithful():
    assert _fails(_Mutant(attention_backward=_backward_variant()),
                  [pin_backward_finite_differences, pin_backward_autograd]) == []


def test_planted_backward_drops_softmax_correction():
    assert _fails(_Mutant(attention_backward=_backward_variant(drop_d=True)),
                  [pin_backward_finite_differences])


def test_planted_backward_misses_gqa_sum():
    assert _fails(_Mutant(attention_backward=_backward_variant(last_head_only=True)),
                  [pin_backward_finite_differences, pin_backward_autograd])


def test_planted_backward_rotates_forward():
    assert _fails(_Mutant(attention_backward=_backward_variant(forward_rotation=True)),
                  [pin_backward_finite_differences, pin_backward_autograd])


def test_planted_paged_offset_swapped():
    def bad(q, k_pages, v_pages, block_table, seq_lens, page_size, scale=None):
        kp, vp = np.asarray(k_pages, np.float64), np.asarray(v_pages, np.float64)
        bt = np.asarray(block_table).astype(np.int64)
        lens = [int(x) for x in seq_lens]
        B, Hkv, d = len(lens), kp.shape[1], kp.shape[3]
        kc = np.zeros((B, Hkv, max(lens), d))
        vc = np.zeros((B, Hkv, max(lens), d))
        n_lp = bt.shape[1]
        for b, L in enumerate(lens):
            for t in range(L):
                page, off = bt[b, t % n_lp], t // n_lp  # page and offset taken the wrong way
                if off >= page_size:
                    off = page_size - 1
                kc[b, :, t] = kp[page, :, off]
                vc[b, :, t] = vp[page, :, off]
        return OA.decode(q, kc, vc, lens, scale=scale)
    assert _fails(_Mutant(decode_paged=bad), [pin_decode_paged_equals_contiguous])


def test_planted_scale_from_value_width():
    """The default scale taken from v's width instead of the keys' fails a pin."""
    assert _fails(_Mutant(scale_from_v=True), [pin_value_width])


def test_planted_cache_append_position_ignores_offset():
    """Keys rotated at t instead of cache_lens[b] + t fail a pin."""
    def bad(k_new, v_new, k_cache, v_cache, cache_lens, *, rope_base=0.0,
            rope_layout="split_half", operand_dtype=None):
        kc = np.array(k_cache, dtype=np.float64)
        vc = np.array(v_cache, dtype=np.float64)
        kn = np.asarray(k_new, dtype=np.float64)
        Tn = kn.shape[2]
        for b, L in enumerate(cache_lens):
            kr = OA.rope_rotate(kn[b], np.arange(Tn), rope_base, rope_layout) if rope_base > 0 else kn[b]
            kc[b, :, L:L + Tn] = OA.round_to(kr, operand_dtype)
            vc[b, :, L:L + Tn] = np.asarray(v_new, dtype=np.float64)[b]
        return kc, vc
    assert _fails(_Mutant(cache_append=bad), [pin_cache_append_positions])


def test_planted_paged_append_offset_swapped():
    """Page and offset swapped in the paged append fail a pin."""
    def bad(k_new, v_new, k_pages, v_pages, block_table, cache_lens, page_size, *,
            rope_base=0.0, rope_layout="split_half", operand_dtype=None):
        kp = np.array(k_pages, dtype=np.float64)
        vp = np.array(v_pages, dtype=np.float64)
        kn = np.asarray(k_new, dtype=np.float64)
        vn = np.asarray(v_new, dtype=np.float64)
        bt = np.asarray(block_table)
        for b, L in enumerate(cache_lens):
            kr = OA.rope_rotate(kn[b], L + np.arange(kn.shape[2]), rope_base, rope_layout)
            for t in range(kn.shape[2]):
                r = L + t
                page, off = bt[b, r % page_size], r // page_size
                kp[page, :, off] = kr[:, t]
                vp[page, :, off] = vn[b, :, t]
        return kp, vp
    assert _fails(_Mutant(cache_append_paged=bad), [pin_cache_append_paged_equals_contiguous])


def test_planted_paged_prefill_positions_ignore_prefix():
    """Queries rotated at i instead of cache_lens[b] + i in the paged prefill fail a pin."""
    def bad(q, k_pages, v_pages, block_table, cache_lens, page_size, *, causal=True,
            rope_base=0.0, scale=None, rope_layout="split_half", operand_dtype=None, lse=False):
        qz = np.asarray(q, np.float64)
        Tq = qz.shape[2]
        res = []
        for b, L in enumerate(cache_lens):
            qr = OA.round_to(OA.rope_rotate(qz[b:b + 1], np.arange(Tq), rope_base, rope_layout),
                             operand_dtype)
            o_b = OA.prefill_paged(qr, k_pages, v_pages, block_table[b:b + 1], [L], page_size,
                                   causal=causal, rope_base=0.0, scale=scale, lse=lse)
            res.append(o_b)
        if lse:
            return (np.concatenate([r[0] for r in res]), np.concatenate([r[1] for r in res]))
        return np.concatenate(res)
    assert _fails(_Mutant(prefill_paged=bad), [pin_prefill_paged_equals_chunk])


def _lse_variant(log2=False, unscaled=False, no_mask=False):
    """The oracle's log-sum-exp with one planted mistake."""
    def lse(q, k, *, causal=True, rope_base=0.0, scale=None, rope_layout="split_half",
            operand_dtype=None, q_offset=0):
        q, k = np.asarray(q, np.float64), np.asarray(k, np.float64)
        B, Hq, T, d = q.shape
        Tk = k.shape[2]
        sc = 1 / math.sqrt(d) if (scale is None or scale <= 0) else scale
        if unscaled:
            sc = 1.0
        if rope_base > 0:
            q = OA.round_to(OA.rope_rotate(q, q_offset + np.arange(T), rope_base, rope_layout),
                            operand_dtype)
            k = OA.round_to(OA.rope_rotate(k, np.arange(Tk), rope_base, rope_layout), operand_dtype)
        kf = OA.expand_kv_heads(k, Hq)
        mask = OA.causal_additive_mask(T, Tk, q_offset) if (causal and not no_mask) else 0.0
        out = np.empty((B, Hq, T))
        for b in range(B):
            for h in range(Hq):
                s = q[b, h] @ kf[b, h].T * sc + mask
                m = np.max(s, axis=-1)
                z = np.sum(np.exp(s - m[:, None]), axis=-1)
                out[b, h] = (m + np.log2(z)) if log2 else (m + np.log(z))
        return out
    return lse


def test_lse_variant_helper_is_faithful():
    assert _fails(_Mutant(attention_lse=_lse_variant()), LSE_PINS) == []


def test_planted_lse_log2():
    assert _fails(_Mutant(attention_lse=_lse_variant(log2=True)), LSE_PINS)


def test_planted_lse_unscaled():
    assert _fails(_Mutant(attention_lse=_lse_variant(unscaled=True)), LSE_PINS)


def test_planted_lse_ignores_mask():
    assert _fails(_Mutant(attention_lse=_lse_variant(no_mask=True)), LSE_PINS)
