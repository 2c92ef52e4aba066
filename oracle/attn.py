"""Plain float64 definition of causal GQA attention. TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs may use this module.  It is slow on purpose: every step is the
textbook definition, with no tiling, fusion, online softmax or reordering.

Sources (page title, then section):
  * "The Transformer architecture" (cooking-agi), "Scaled dot-product attention":
    Attention(Q,K,V) = softmax(Q K^T / sqrt(d_k)) V, per query
    o_i = sum_j alpha_ij v_j with alpha_ij = exp(q_i.k_j/sqrt(d_k)) / sum_j' ...
  * "Transformer" (ai-notes), "Scaled dot-product attention" and "What is the
    causal mask?": Attn(Q,K,V;M) = softmax(Q K^T / sqrt(d_k) + M) V with the
    additive mask M[t,s] = 0 for s <= t and -inf for s > t.
  * "Transformer Math and Implementation Deep Dive", "Attention Shapes",
    "Attention Equation", "Causal Masking": q [B, n_q_heads, T, d_head],
    k/v [B, n_kv_heads, T, d_head]; GQA maps KV heads across query-head groups;
    scores[i, j] = -inf if j > i.
  * "The Transformer architecture", "Now: RoPE": rotation of q and k (never v)
    by R_m per channel pair; the split-half pairing (channel i with i + d/2).
  * "Transformer" (ai-notes), "RoPE (Rotary Positional Embedding)": adjacent
    pairs (2i, 2i+1) with angle theta_i(pos) = pos * 10000^(-2i/d_head); the
    base 10000 is the ``rope_base`` argument here.
  * "The Transformer architecture", "What else the modern decoder-only model
    changed": each group of n_rep query heads shares one K/V head.
  * "The Transformer architecture", "Hands-on": with a cache, the query at
    position p sees keys 0..p, the current token included.  The same holds for
    a chunk of Tq new queries after a cache prefix of length q_offset: query i
    sits at position q_offset + i, is rotated at that position, and sees keys
    0..q_offset+i (the cache plus the chunk's own causal part).
  * "Transformer Math and Implementation Deep Dive", "Attention Equation"
    (cross-attention): with no causal mask, Tq and Tk need not be equal.

Readings where the pages leave a step open:
  * RoPE frequencies theta_i = base^(-2i/d), i = 0..d/2-1, positions from 0.
  * The rotated q and k are rounded to the input dtype (round-to-nearest-even)
    before the dot product, as the pages' ``apply_rope`` returns a tensor of the
    input's dtype; everything after that is float64.
  * Query head h reads KV head h // (Hq/Hkv) (contiguous groups).
  * A row with no visible key (only possible in decode with length 0) has
    output 0.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "softmax_rows", "rope_inv_freq", "rope_cos_sin", "rope_rotate", "round_to",
    "round_to_bf16", "expand_kv_heads", "causal_additive_mask", "attention_scores",
    "attention", "attention_rows", "attention_lse", "attention_backward", "decode",
    "decode_paged", "decode_step", "merge_partials", "split_partials", "rope_rotate_transpose",
    "cache_append", "cache_append_paged", "prefill_paged"]

_BF16_MAX = float.fromhex("0x1.fep127")


def softmax_rows(z):
    """Row softmax over the last axis: e^{z_i} / sum_j e^{z_j}.

    "The Transformer architecture", "Softmax is a differentiable allocation":
    applied row by row over the last dimension of the score matrix.  The row
    maximum is subtracted first (exact in real arithmetic).  A row that is
    entirely -inf gives all-zero weights.
    """
    z = np.asarray(z, dtype=np.float64)
    m = np.max(z, axis=-1, keepdims=True)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    e = np.exp(z - m_safe)  # exp(-inf) == 0 exactly
    s = np.sum(e, axis=-1, keepdims=True)
    out = np.where(finite, e / np.where(s > 0, s, 1.0), 0.0)
    return out


def rope_inv_freq(d: int, base: float):
    """theta_i = base^(-2i/d) for i = 0..d/2-1 ("Transformer" (ai-notes), RoPE section)."""
    i = np.arange(d // 2, dtype=np.float64)
    return np.power(float(base), -(2.0 * i) / float(d))


def rope_cos_sin(positions, d: int, base: float):
    """cos and sin of the angle pos * theta_i, in float64; shape [len(positions), d/2]."""
    pos = np.asarray(positions, dtype=np.float64)
    ang = np.outer(pos, rope_inv_freq(d, base))
    return np.cos(ang), np.sin(ang)


def rope_rotate(x, positions, base: float, layout: str = "split_half"):
    """Rotate each channel pair of x[..., T, d] by R_pos.

    Pair (a, b) becomes (a cos - b sin, a sin + b cos).  ``split_half`` pairs
    channel i with i + d/2 ("The Transformer architecture", "Now: RoPE");
    ``adjacent`` pairs 2i with 2i+1 ("Transformer" (ai-notes), RoPE section).
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    c, s = rope_cos_sin(positions, d, base)
    out = np.empty_like(x)
    if layout == "split_half":
        a, b = x[..., : d // 2], x[..., d // 2:]
        out[..., : d // 2] = a * c - b * s
        out[..., d // 2:] = a * s + b * c
    elif layout == "adjacent":
        a, b = x[..., 0::2], x[..., 1::2]
        out[..., 0::2] = a * c - b * s
        out[..., 1::2] = a * s + b * c
    else:
        raise ValueError(f"unknown RoPE layout {layout!r}")
    return out


def round_to_bf16(x):
    """Round float64 values to the nearest bfloat16 (ties to even), returned as float64.

    bfloat16 keeps 8 significant bits and the float32 exponent range; values
    below 2^-126 are on the subnormal grid of step 2^-133.
    """
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(invalid="ignore", over="ignore"):
        _, e = np.frexp(x)
        e = np.maximum(e, -125)
        y = np.ldexp(np.rint(np.ldexp(x, 8 - e)), e - 8)
        y = np.where(np.abs(y) > _BF16_MAX, np.copysign(np.inf, y), y)
    return np.where(np.isfinite(x), y, x)


def round_to(x, dtype):
    """Round to the operand dtype: None (keep float64), 'f32' or 'bf16'."""
    if dtype is None:
        return np.asarray(x, dtype=np.float64)
    if dtype == "f32":
        return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)
    if dtype == "bf16":
        return round_to_bf16(x)
    raise ValueError(f"unknown dtype {dtype!r}")


def expand_kv_heads(kv, n_q_heads: int):
    """Repeat KV heads so query head h reads KV head h // (Hq/Hkv).

    kv has the head axis at position -3 ([..., Hkv, T, d]).
    """
    kv = np.asarray(kv, dtype=np.float64)
    hkv = kv.shape[-3]
    if n_q_heads % hkv != 0:
        raise ValueError("n_q_heads must be a multiple of n_kv_heads")
    return np.repeat(kv, n_q_heads // hkv, axis=-3)


def causal_additive_mask(tq: int, tk: int, q_offset: int = 0):
    """M[i, j] = 0 if key j <= query position (q_offset + i), else -inf."""
    i = np.arange(tq)[:, None] + int(q_offset)
    j = np.arange(tk)[None, :]
    return np.where(j > i, -np.inf, 0.0)


def attention_scores(q, k, scale: float):
    """(Q K^T) * scale for q [..., Tq, d], k [..., Tk, d]."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    return (q @ np.swapaxes(k, -1, -2)) * float(scale)


def _default_scale(d, scale):
    return 1.0 / math.sqrt(d) if (scale is None or scale <= 0) else float(scale)


def _rotated(x, base, layout, operand_dtype, positions):
    if base is None or base <= 0:
        return np.asarray(x, dtype=np.float64)
    return round_to(rope_rotate(x, positions, base, layout), operand_dtype)


def attention(q, k, v, *, causal=True, rope_base=0.0, scale=None,
              rope_layout="split_half", operand_dtype=None, q_offset=0):
    """Full prefill output [B, Hq, Tq, d] in float64.

    q [B, Hq, Tq, d]; k, v [B, Hkv, Tk, d].  Query i sits at position
    q_offset + i, key j at position j.  Steps: upcast; RoPE on q and k at
    those positions, rounded to ``operand_dtype``; GQA repetition of K/V;
    S = Q K^T * scale; S + M (key j visible iff j <= q_offset + i when
    causal); row softmax; P V.  Loops over (b, h) to bound memory.
    """
    q = np.asarray(_as_np(q), dtype=np.float64)
    k = np.asarray(_as_np(k), dtype=np.float64)
    v = np.asarray(_as_np(v), dtype=np.float64)
    B, Hq, T, d = q.shape
    Tk = k.shape[2]
    sc = _default_scale(d, scale)
    qr = _rotated(q, rope_base, rope_layout, operand_dtype, int(q_offset) + np.arange(T))
    kr = _rotated(k, rope_base, rope_layout, operand_dtype, np.arange(Tk))
    kf = expand_kv_heads(kr, Hq)
    vf = expand_kv_heads(v, Hq)
    mask = causal_additive_mask(T, Tk, q_offset) if causal else np.zeros((T, Tk))
    out = np.empty((B, Hq, T, v.shape[-1]), dtype=np.float64)
    for b in range(B):
        for h in range(Hq):
            s = attention_scores(qr[b, h], kf[b, h], sc) + mask
            out[b, h] = softmax_rows(s) @ vf[b, h]
    return out


def attention_lse(q, k, *, causal=True, rope_base=0.0, scale=None,
                  rope_layout="split_half", operand_dtype=None, q_offset=0):
    """Natural-log log-sum-exp of each masked score row, [B, Hq, Tq]."""
    q = np.asarray(_as_np(q), dtype=np.float64)
    k = np.asarray(_as_np(k), dtype=np.float64)
    B, Hq, T, d = q.shape
    Tk = k.shape[2]
    sc = _default_scale(d, scale)
    qr = _rotated(q, rope_base, rope_layout, operand_dtype, int(q_offset) + np.arange(T))
    kf = expand_kv_heads(_rotated(k, rope_base, rope_layout, operand_dtype, np.arange(Tk)), Hq)
    mask = causal_additive_mask(T, Tk, q_offset) if causal else np.zeros((T, Tk))
    out = np.empty((B, Hq, T), dtype=np.float64)
    for b in range(B):
        for h in range(Hq):
            s = attention_scores(qr[b, h], kf[b, h], sc) + mask
            m = np.max(s, axis=-1)
            out[b, h] = m + np.log(np.sum(np.exp(s - m[:, None]), axis=-1))
    return out


def attention_rows(q, k, v, b: int, h: int, rows, *, causal=True, rope_base=0.0,
                   scale=None, rope_layout="split_half", operand_dtype=None, q_offset=0):
    """Output rows ``rows`` of head h, batch b: [len(rows), d] float64.

    Same definition as ``attention`` restricted to a subset of query rows, for
    workloads whose full T x T score matrix does not fit in host memory.
    q/k/v may be torch CPU tensors or numpy arrays of the full problem.
    """
    rows = np.asarray(rows, dtype=np.int64)
    Hq, T, d = q.shape[1], q.shape[2], q.shape[3]
    Hkv, Tk = k.shape[1], k.shape[2]
    g = h // (Hq // Hkv)
    qb = np.asarray(_as_np(q[b, h]), dtype=np.float64)[rows]
    kb = np.asarray(_as_np(k[b, g]), dtype=np.float64)
    vb = np.asarray(_as_np(v[b, g]), dtype=np.float64)
    sc = _default_scale(d, scale)
    pos = int(q_offset) + rows
    qr = _rotated(qb, rope_base, rope_layout, operand_dtype, pos)
    kr = _rotated(kb, rope_base, rope_layout, operand_dtype, np.arange(Tk))
    s = attention_scores(qr, kr, sc)
    if causal:
        s = s + np.where(np.arange(Tk)[None, :] > pos[:, None], -np.inf, 0.0)
    return softmax_rows(s) @ vb


def decode(q, k_cache, v_cache, seq_lens, scale=None):
    """KV-cache decode: one query per (b, q-head) over cache rows 0..L_b-1.

    q [B, Hq, 1, d] and the cache [B, Hkv, Lmax, d] are already in rotated
    space; the query sits at position L_b - 1 and every cached row, the
    current token's included, is visible.  Rows >= L_b are never read.
    """
    B, Hq, _, d = q.shape
    sc = _default_scale(d, scale)
    out = np.zeros((B, Hq, 1, v_cache.shape[-1]), dtype=np.float64)
    for b in range(B):
        L = int(seq_lens[b])
        if L <= 0:
            continue
        kb = expand_kv_heads(np.asarray(_as_np(k_cache[b, :, :L]), dtype=np.float64), Hq)
        vb = expand_kv_heads(np.asarray(_as_np(v_cache[b, :, :L]), dtype=np.float64), Hq)
        qb = np.asarray(_as_np(q[b, :, 0]), dtype=np.float64)
        s = np.einsum("hd,hld->hl", qb, kb) * sc
        out[b, :, 0] = np.einsum("hl,hld->hd", softmax_rows(s), vb)
    return out


def decode_paged(q, k_pages, v_pages, block_table, seq_lens, page_size: int, scale=None):
    """Decode over a paged cache: k_pages, v_pages [num_pages, Hkv, page_size, d];
    row t of sequence b lives in page block_table[b][t // page_size] at offset
    t % page_size.  The pages of each sequence are gathered into a contiguous
    cache and ``decode`` applies."""
    kp = np.asarray(_as_np(k_pages), dtype=np.float64)
    vp = np.asarray(_as_np(v_pages), dtype=np.float64)
    bt = np.asarray(_as_np(block_table)).astype(np.int64)
    lens = [int(x) for x in np.asarray(_as_np(seq_lens)).reshape(-1)]
    B = len(lens)
    Hkv, d = kp.shape[1], kp.shape[3]
    Lmax = max(1, max(lens))
    kc = np.zeros((B, Hkv, Lmax, d))
    vc = np.zeros((B, Hkv, Lmax, d))
    for b, L in enumerate(lens):
        for t in range(L):
            page, off = bt[b, t // page_size], t % page_size
            kc[b, :, t] = kp[page, :, off]
            vc[b, :, t] = vp[page, :, off]
    return decode(q, kc, vc, lens, scale=scale)


def decode_step(q_new, k_new, v_new, k_cache, v_cache, cache_lens, *, rope_base=0.0,
                rope_layout="split_half", scale=None, operand_dtype=None):
    """One decode step with the new token's K/V appended to the cache first.

    q_new [B, Hq, 1, d], k_new / v_new [B, Hkv, 1, d] are the new token's
    projections, not rotated; the cache [B, Hkv, Lmax, d] holds rotated keys.
    For sequence b the new token sits at position p = cache_lens[b] ("The
    Transformer architecture", "Hands-on": the cache grows by one row per
    generated token and the query at cache.pos sees keys 0..cache.pos): q and k
    are rotated at p and rounded to ``operand_dtype``, k and v are written to
    cache row p, and the query attends to rows 0..p.  Returns (out, k_cache',
    v_cache') with the caches as new float64 arrays.
    """
    q_new = np.asarray(_as_np(q_new), dtype=np.float64)
    k_new = np.asarray(_as_np(k_new), dtype=np.float64)
    v_new = np.asarray(_as_np(v_new), dtype=np.float64)
    kc = np.array(_as_np(k_cache), dtype=np.float64)
    vc = np.array(_as_np(v_cache), dtype=np.float64)
    B, Hq, _, d = q_new.shape
    qr = np.empty_like(q_new)
    lens = [int(x) for x in np.asarray(_as_np(cache_lens)).reshape(-1)]
    for b, pos in enumerate(lens):
        at = np.array([pos])
        qr[b] = _rotated(q_new[b], rope_base, rope_layout, operand_dtype, at)
        kc[b, :, pos] = _rotated(k_new[b], rope_base, rope_layout, operand_dtype, at)[:, 0]
        vc[b, :, pos] = v_new[b, :, 0]
    out = decode(qr, kc, vc, [L + 1 for L in lens], scale=scale)
    return out, kc, vc


def cache_append(k_new, v_new, k_cache, v_cache, cache_lens, *, rope_base=0.0,
                 rope_layout="split_half", operand_dtype=None):
    """Append Tn tokens per sequence to contiguous caches [B, Hkv, Lmax, d].

    Token t of sequence b sits at position p = cache_lens[b] + t ("The
    Transformer architecture", "Hands-on": the cache grows by one row per
    token, at cache.pos); its key is rotated at p (RoPE on keys, never on
    values: same page, "Now: RoPE") and rounded to ``operand_dtype``, and key
    and value are written to row p.  Returns the new caches as float64 arrays.
    """
    k_new = np.asarray(_as_np(k_new), dtype=np.float64)
    v_new = np.asarray(_as_np(v_new), dtype=np.float64)
    kc = np.array(_as_np(k_cache), dtype=np.float64)
    vc = np.array(_as_np(v_cache), dtype=np.float64)
    Tn = k_new.shape[2]
    lens = [int(x) for x in np.asarray(_as_np(cache_lens)).reshape(-1)]
    for b, L in enumerate(lens):
        pos = L + np.arange(Tn)
        kc[b, :, L:L + Tn] = _rotated(k_new[b], rope_base, rope_layout, operand_dtype, pos)
        vc[b, :, L:L + Tn] = v_new[b]
    return kc, vc


def cache_append_paged(k_new, v_new, k_pages, v_pages, block_table, cache_lens, page_size: int,
                       *, rope_base=0.0, rope_layout="split_half", operand_dtype=None):
    """``cache_append`` into paged caches [num_pages, Hkv, page_size, d]: row r of
    sequence b lives in page block_table[b][r // page_size] at offset r % page_size.
    Returns the new page pools as float64 arrays."""
    k_new = np.asarray(_as_np(k_new), dtype=np.float64)
    v_new = np.asarray(_as_np(v_new), dtype=np.float64)
    kp = np.array(_as_np(k_pages), dtype=np.float64)
    vp = np.array(_as_np(v_pages), dtype=np.float64)
    bt = np.asarray(_as_np(block_table)).astype(np.int64)
    Tn = k_new.shape[2]
    lens = [int(x) for x in np.asarray(_as_np(cache_lens)).reshape(-1)]
    for b, L in enumerate(lens):
        kr = _rotated(k_new[b], rope_base, rope_layout, operand_dtype, L + np.arange(Tn))
        for t in range(Tn):
            r = L + t
            page, off = bt[b, r // page_size], r % page_size
            kp[page, :, off] = kr[:, t]
            vp[page, :, off] = v_new[b, :, t]
    return kp, vp


def prefill_paged(q, k_pages, v_pages, block_table, cache_lens, page_size: int, *, causal=True,
                  rope_base=0.0, scale=None, rope_layout="split_half", operand_dtype=None,
                  lse=False):
    """Chunk prefill over a paged cache of rotated keys ("The Transformer
    architecture", "Hands-on"): for sequence b with L = cache_lens[b], cache rows
    0..L+Tq-1 (the prefix, then the chunk's own rows) are gathered from the pages
    (row t in page block_table[b][t // page_size] at offset t % page_size); query
    i is rotated at position L + i (rounded to ``operand_dtype``), the keys are used
    as stored, and the attention definition with that query offset applies.
    Returns out [B, Hq, Tq, d] (and the natural-log lse [B, Hq, Tq] with lse=True).
    """
    q = np.asarray(_as_np(q), dtype=np.float64)
    kp = np.asarray(_as_np(k_pages), dtype=np.float64)
    vp = np.asarray(_as_np(v_pages), dtype=np.float64)
    bt = np.asarray(_as_np(block_table)).astype(np.int64)
    lens = [int(x) for x in np.asarray(_as_np(cache_lens)).reshape(-1)]
    B, Hq, Tq, d = q.shape
    Hkv = kp.shape[1]
    out = np.empty((B, Hq, Tq, vp.shape[-1]), dtype=np.float64)
    lses = np.empty((B, Hq, Tq), dtype=np.float64)
    for b, L in enumerate(lens):
        Tk = L + Tq
        kc = np.empty((1, Hkv, Tk, d))
        vc = np.empty((1, Hkv, Tk, vp.shape[-1]))
        for t in range(Tk):
            page, off = bt[b, t // page_size], t % page_size
            kc[0, :, t] = kp[page, :, off]
            vc[0, :, t] = vp[page, :, off]
        qr = _rotated(q[b:b + 1], rope_base, rope_layout, operand_dtype, L + np.arange(Tq))
        out[b] = attention(qr, kc, vc, causal=causal, rope_base=0.0, scale=scale, q_offset=L)[0]
        if lse:
            lses[b] = attention_lse(qr, kc, causal=causal, rope_base=0.0, scale=scale,
                                    q_offset=L)[0]
    return (out, lses) if lse else out


def rope_rotate_transpose(x, positions, base: float, layout: str = "split_half"):
    """R_pos^T x, the transpose (= inverse) of ``rope_rotate``'s rotation: the
    chain rule applies it to a gradient flowing back through RoPE.

    Pair (a, b) becomes (a cos + b sin, -a sin + b cos).
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    c, s = rope_cos_sin(positions, d, base)
    out = np.empty_like(x)
    if layout == "split_half":
        a, b = x[..., : d // 2], x[..., d // 2:]
        out[..., : d // 2] = a * c + b * s
        out[..., d // 2:] = -a * s + b * c
    elif layout == "adjacent":
        a, b = x[..., 0::2], x[..., 1::2]
        out[..., 0::2] = a * c + b * s
        out[..., 1::2] = -a * s + b * c
    else:
        raise ValueError(f"unknown RoPE layout {layout!r}")
    return out


def attention_backward(q, k, v, dout, *, causal=True, rope_base=0.0, scale=None,
                       rope_layout="split_half", operand_dtype=None, q_offset=0):
    """Gradients (dq, dk, dv) of sum(out * dout) for out = attention(q, k, v, ...).

    The derivative of the definition above, written out (float64):
      P = softmax(S + M),  S = scale * Qr Kr^T,  O = P V          (per query head)
      dV_g  = sum over the heads h of group g of P_h^T dO_h
      dP    = dO V^T;  dS = P o (dP - D),  D_i = sum_c dO_ic O_ic  (softmax Jacobian)
      dQr   = scale * dS Kr;  dKr_g = scale * sum_h dS_h^T Qr_h
      dq    = R^T dQr,  dk = R^T dKr   (RoPE is a rotation: its Jacobian is R)
    Rounding of the rotated operands to ``operand_dtype`` is part of the forward;
    the backward treats it as the identity (its derivative is zero almost
    everywhere, which no training step uses), so the gradients are those of the
    unrounded function evaluated at the rounded operands.
    """
    q = np.asarray(_as_np(q), dtype=np.float64)
    k = np.asarray(_as_np(k), dtype=np.float64)
    v = np.asarray(_as_np(v), dtype=np.float64)
    do = np.asarray(_as_np(dout), dtype=np.float64)
    B, Hq, T, d = q.shape
    Hkv, Tk = k.shape[1], k.shape[2]
    rep = Hq // Hkv
    sc = _default_scale(d, scale)
    qpos = int(q_offset) + np.arange(T)
    kpos = np.arange(Tk)
    qr = _rotated(q, rope_base, rope_layout, operand_dtype, qpos)
    kr = _rotated(k, rope_base, rope_layout, operand_dtype, kpos)
    mask = causal_additive_mask(T, Tk, q_offset) if causal else np.zeros((T, Tk))
    dqr = np.zeros_like(qr)
    dkr = np.zeros_like(kr)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(Hq):
            g = h // rep
            p = softmax_rows(attention_scores(qr[b, h], kr[b, g], sc) + mask)
            o = p @ v[b, g]
            dv[b, g] += p.T @ do[b, h]
            dp = do[b, h] @ v[b, g].T
            dsc = p * (dp - np.sum(do[b, h] * o, axis=-1, keepdims=True))
            dqr[b, h] = sc * (dsc @ kr[b, g])
            dkr[b, g] += sc * (dsc.T @ qr[b, h])
    if rope_base is not None and rope_base > 0:
        dq = rope_rotate_transpose(dqr, qpos, rope_base, rope_layout)
        dk = rope_rotate_transpose(dkr, kpos, rope_base, rope_layout)
    else:
        dq, dk = dqr, dkr
    return dq, dk, dv


def split_partials(s, v, bounds):
    """Per-split (max, sum, unnormalised output) of one score row s [L] over v [L, d].

    Split j covers keys bounds[j]..bounds[j+1]-1.  An empty split gives
    (-inf, 0, 0).  This is the softmax split along the key axis that a
    split-KV decode computes; ``merge_partials`` puts it back together.
    """
    s = np.asarray(s, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    ms, ls, os = [], [], []
    for a, e in zip(bounds[:-1], bounds[1:]):
        if e <= a:
            ms.append(-np.inf)
            ls.append(0.0)
            os.append(np.zeros(v.shape[-1]))
            continue
        m = np.max(s[a:e])
        p = np.exp(s[a:e] - m)
        ms.append(m)
        ls.append(np.sum(p))
        os.append(p @ v[a:e])
    return np.array(ms), np.array(ls), np.array(os)


def merge_partials(ms, ls, os):
    """Merge split softmax partials: m = max m_j, l = sum l_j e^{m_j - m},
    o = sum o_j e^{m_j - m} / l.  Exact identity of the softmax (real arithmetic)."""
    ms = np.asarray(ms, dtype=np.float64)
    m = np.max(ms)
    if not np.isfinite(m):
        return np.zeros(np.asarray(os).shape[-1])
    w = np.exp(ms - m)
    l_tot = np.sum(np.asarray(ls) * w)
    return (w[:, None] * np.asarray(os, dtype=np.float64)).sum(axis=0) / l_tot


def _as_np(t):
    if hasattr(t, "detach"):
        return t.detach().float().numpy() if t.dtype != _torch_f64() else t.detach().numpy()
    return t


def _torch_f64():
    import torch
    return torch.float64
