"""Scalar-loop attention for tiny inputs. TEST INFRASTRUCTURE.

Written separately from ``oracle.attn`` (it imports nothing from it) to
brute-force-check it: Python floats, ``math.exp``/``math.cos``/``math.sin`` and
explicit loops over batch, head, query, key and channel, following the
per-query form of "The Transformer architecture" (cooking-agi), section
"Scaled dot-product attention":

    alpha_ij = exp(q_i . k_j / sqrt(d_k)) / sum_j' exp(q_i . k_j' / sqrt(d_k)),
    o_i = sum_j alpha_ij v_j,

where keys j > i are left out of both sums under the causal mask (their weight
is exactly zero: "Grasping Codes and Math 02", "Why Fill with Negative
Infinity?").  RoPE follows "Transformer" (ai-notes), section "RoPE (Rotary
Positional Embedding)": pair p of channels is turned by the angle
pos * base^(-2p/d).  Query head h reads KV head floor(h / (Hq/Hkv)).
"""
from __future__ import annotations

import math
from fractions import Fraction

__all__ = ["naive_attention", "naive_lse", "naive_round_bf16", "naive_decode"]


def naive_round_bf16(x: float) -> float:
    """Nearest bfloat16 to x, ties to even, by exact rational arithmetic."""
    if x == 0.0 or math.isnan(x) or math.isinf(x):
        return x
    _, e = math.frexp(x)
    e = max(e, -125)
    step = Fraction(2) ** (e - 8)
    r = Fraction(x) / step
    n = math.floor(r)
    frac = r - n
    if frac > Fraction(1, 2) or (frac == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return float(n * step)


def _rot(vec, pos, base, layout, rnd):
    d = len(vec)
    out = list(vec)
    for p in range(d // 2):
        ang = pos * (base ** (-(2.0 * p) / d))
        c, s = math.cos(ang), math.sin(ang)
        if layout == "split_half":
            i, j = p, p + d // 2
        else:
            i, j = 2 * p, 2 * p + 1
        a, b = vec[i], vec[j]
        out[i] = a * c - b * s
        out[j] = a * s + b * c
    if rnd is not None:
        out = [rnd(x) for x in out]
    return out


def naive_attention(q, k, v, causal=True, rope_base=0.0, scale=None,
                    rope_layout="split_half", round_bf16=False, q_offset=0):
    """q [B][Hq][Tq][d], k/v [B][Hkv][Tk][d] as nested lists; returns nested lists.

    Query i sits at position q_offset + i (RoPE angle and causal limit)."""
    B, Hq, T, d = len(q), len(q[0]), len(q[0][0]), len(q[0][0][0])
    Hkv = len(k[0])
    Tk = len(k[0][0])
    rep = Hq // Hkv
    sc = (1.0 / math.sqrt(d)) if (scale is None or scale <= 0) else scale
    rnd = naive_round_bf16 if round_bf16 else None
    out = []
    for b in range(B):
        ob = []
        for h in range(Hq):
            g = h // rep
            if rope_base > 0:
                qs = [_rot(q[b][h][t], q_offset + t, rope_base, rope_layout, rnd)
                      for t in range(T)]
                ks = [_rot(k[b][g][t], t, rope_base, rope_layout, rnd) for t in range(Tk)]
            else:
                qs = [list(map(float, q[b][h][t])) for t in range(T)]
                ks = [list(map(float, k[b][g][t])) for t in range(Tk)]
            vs = v[b][g]
            oh = []
            for i in range(T):
                scores = {}
                for j in range(Tk):
                    if causal and j > q_offset + i:
                        continue
                    dot = 0.0
                    for c in range(d):
                        dot += qs[i][c] * ks[j][c]
                    scores[j] = dot * sc
                mx = max(scores.values())
                w = {j: math.exp(s - mx) for j, s in scores.items()}
                z = sum(w.values())
                row = []
                for c in range(len(vs[0])):
                    acc = 0.0
                    for j, wj in w.items():
                        acc += wj * vs[j][c]
                    row.append(acc / z)
                oh.append(row)
            ob.append(oh)
        out.append(ob)
    return out


def naive_lse(q, k, causal=True, rope_base=0.0, scale=None, rope_layout="split_half",
              round_bf16=False, q_offset=0):
    """Natural log of each query's softmax denominator, nested lists [B][Hq][Tq].

    The softmax of "The Transformer architecture", "Softmax is a differentiable
    allocation" divides by z_i = sum_j exp(s_ij) over the visible keys; this is
    ln z_i, computed as max_j s_ij + ln sum_j exp(s_ij - max_j s_ij) with the
    same scalar loops as ``naive_attention`` (s_ij = q_i . k_j * scale).
    """
    B, Hq, T, d = len(q), len(q[0]), len(q[0][0]), len(q[0][0][0])
    Hkv = len(k[0])
    Tk = len(k[0][0])
    rep = Hq // Hkv
    sc = (1.0 / math.sqrt(d)) if (scale is None or scale <= 0) else scale
    rnd = naive_round_bf16 if round_bf16 else None
    out = []
    for b in range(B):
        ob = []
        for h in range(Hq):
            g = h // rep
            row = []
            for i in range(T):
                if rope_base > 0:
                    qi = _rot(q[b][h][i], q_offset + i, rope_base, rope_layout, rnd)
                else:
                    qi = [float(x) for x in q[b][h][i]]
                s = []
                for j in range(Tk):
                    if causal and j > q_offset + i:
                        continue
                    if rope_base > 0:
                        kj = _rot(k[b][g][j], j, rope_base, rope_layout, rnd)
                    else:
                        kj = [float(x) for x in k[b][g][j]]
                    dot = 0.0
                    for c in range(d):
                        dot += qi[c] * kj[c]
                    s.append(dot * sc)
                mx = max(s)
                z = 0.0
                for x in s:
                    z += math.exp(x - mx)
                row.append(mx + math.log(z))
            ob.append(row)
        out.append(ob)
    return out


def naive_decode(q, k_cache, v_cache, seq_lens, scale=None):
    """q [B][Hq][d] (one query each), caches [B][Hkv][Lmax][d]; rows < seq_lens[b] only."""
    B, Hq, d = len(q), len(q[0]), len(q[0][0])
    Hkv = len(k_cache[0])
    rep = Hq // Hkv
    sc = (1.0 / math.sqrt(d)) if (scale is None or scale <= 0) else scale
    out = []
    for b in range(B):
        L = int(seq_lens[b])
        ob = []
        for h in range(Hq):
            g = h // rep
            if L <= 0:
                ob.append([0.0] * d)
                continue
            s = []
            for j in range(L):
                dot = 0.0
                for c in range(d):
                    dot += q[b][h][c] * k_cache[b][g][j][c]
                s.append(dot * sc)
            mx = max(s)
            w = [math.exp(x - mx) for x in s]
            z = sum(w)
            ob.append([sum(w[j] * v_cache[b][g][j][c] for j in range(L)) / z for c in range(d)])
        out.append(ob)
    return out
