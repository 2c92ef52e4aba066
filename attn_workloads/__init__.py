"""Seeded synthetic inputs for causal GQA attention (prefill and KV-cache decode).

This module holds the workload shapes and the random-number recipe only. It
performs none of the attention arithmetic (no RoPE, no scores, no softmax), so
that the CPU oracle and the CUDA path can share it without sharing any of the
method itself.

Recipe (every workload):
  * ``torch.Generator('cpu').manual_seed(seed)``; values drawn with
    ``torch.randn`` in float32, then cast to the workload dtype with
    round-to-nearest-even (bf16) or kept (fp32).
  * prefill: q [B,Hq,T,d], then k [B,Hkv,T,d], then v [B,Hkv,T,d], drawn in
    that order.  ``qk_mult`` (a power of two) multiplies q and k after the
    cast, which is exact.
  * decode: seq_lens = randint(Lmin, Lmax+1, (B,)) first, then q [B,Hq,1,d],
    then for b = 0..B-1 in order k_b [Hkv,L_b,d] and v_b [Hkv,L_b,d].  Cache
    rows at or beyond seq_lens[b] are filled with NaN so that any read of them
    shows up in the output.

The five named workloads follow the shapes in the pages' statement of the
problem: q [B, n_q_heads, T, d_head], k/v [B, n_kv_heads, T, d_head]
("Transformer Math and Implementation Deep Dive", section "Attention Shapes").
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional

import torch

__all__ = [
    "PrefillWorkload",
    "DecodeWorkload",
    "WORKLOADS",
    "make_prefill_inputs",
    "make_decode_inputs",
    "torch_dtype",
]


@dataclass(frozen=True)
class PrefillWorkload:
    name: str
    B: int
    Hq: int
    Hkv: int
    T: int
    d: int
    dtype: str  # "f32" | "bf16"
    rope_base: float  # <= 0 means no RoPE
    scale: float
    causal: bool = True
    seed: int = 0
    qk_mult: float = 1.0
    rope_layout: str = "split_half"  # "split_half" | "adjacent"

    def flops(self) -> float:
        """Causal attention FLOPs 2*B*Hq*T^2*d (QK^T and PV, halved for the mask)."""
        f = 2.0 * self.B * self.Hq * self.T * self.T * self.d
        return f if self.causal else 2.0 * f

    def with_(self, **kw) -> "PrefillWorkload":
        return replace(self, **kw)


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    Lmax: int
    Lmin: int
    dtype: str = "bf16"
    scale: float = 0.0
    seed: int = 0

    def with_(self, **kw) -> "DecodeWorkload":
        return replace(self, **kw)


@dataclass(frozen=True)
class ChunkWorkload:
    """A chunk of Tq queries at positions q_offset.. against Tk keys (a cached prefix
    plus the chunk's own keys when Tk = q_offset + Tq), or rectangular attention."""
    name: str
    B: int
    Hq: int
    Hkv: int
    Tq: int
    Tk: int
    q_offset: int
    d: int
    dtype: str
    rope_base: float
    scale: float
    causal: bool = True
    seed: int = 0

    def visible_keys(self) -> int:
        """Sum over query rows of the keys each one sees (row i: min(Tk, q_offset + i + 1))."""
        if not self.causal:
            return self.Tq * self.Tk
        rows_short = max(0, min(self.Tq, self.Tk - self.q_offset))  # rows seeing < all keys
        seen = rows_short * (2 * self.q_offset + rows_short + 1) // 2
        return seen + (self.Tq - rows_short) * self.Tk

    def flops(self) -> float:
        """QK^T and PV over the visible (query, key) pairs: 4*d per pair."""
        return 4.0 * self.B * self.Hq * self.d * self.visible_keys()

    def with_(self, **kw) -> "ChunkWorkload":
        return replace(self, **kw)


WORKLOADS = {
    "tiny_f32": PrefillWorkload("tiny_f32", B=1, Hq=2, Hkv=2, T=64, d=16, dtype="f32",
                                rope_base=10000.0, scale=1.0 / math.sqrt(16)),
    "gpt2_bf16": PrefillWorkload("gpt2_bf16", B=8, Hq=12, Hkv=12, T=1024, d=64,
                                 dtype="bf16", rope_base=0.0, scale=1.0 / 8.0),
    "llama_gqa_bf16": PrefillWorkload("llama_gqa_bf16", B=4, Hq=32, Hkv=8, T=4096, d=128,
                                      dtype="bf16", rope_base=10000.0,
                                      scale=1.0 / math.sqrt(128)),
    "llama_gqa_bf16_x4": PrefillWorkload("llama_gqa_bf16_x4", B=4, Hq=32, Hkv=8, T=4096,
                                         d=128, dtype="bf16", rope_base=10000.0,
                                         scale=1.0 / math.sqrt(128), seed=1, qk_mult=4.0),
    "long_gqa_bf16": PrefillWorkload("long_gqa_bf16", B=1, Hq=32, Hkv=8, T=32768, d=128,
                                     dtype="bf16", rope_base=500000.0,
                                     scale=1.0 / math.sqrt(128)),
    # the last quarter of the llama_gqa_bf16 sequence as one chunk after a 3072-token cache
    "llama_chunk_bf16": ChunkWorkload("llama_chunk_bf16", B=4, Hq=32, Hkv=8, Tq=1024, Tk=4096,
                                      q_offset=3072, d=128, dtype="bf16", rope_base=10000.0,
                                      scale=1.0 / math.sqrt(128)),
    # cross / rectangular attention: 1024 queries against 4096 keys, no mask, no RoPE
    "llama_cross_bf16": ChunkWorkload("llama_cross_bf16", B=4, Hq=32, Hkv=8, Tq=1024, Tk=4096,
                                      q_offset=0, d=128, dtype="bf16", rope_base=0.0,
                                      scale=1.0 / math.sqrt(128), causal=False),
    "decode_bf16": DecodeWorkload("decode_bf16", B=64, Hq=32, Hkv=8, d=128, Lmax=8192,
                                  Lmin=512, dtype="bf16", scale=1.0 / math.sqrt(128)),
}


def torch_dtype(name: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def make_prefill_inputs(w: PrefillWorkload, seed: Optional[int] = None):
    """Return CPU tensors (q, k, v) in the workload dtype, contiguous."""
    g = _gen(w.seed if seed is None else seed)
    dt = torch_dtype(w.dtype)
    q = torch.randn(w.B, w.Hq, w.T, w.d, generator=g, dtype=torch.float32).to(dt)
    k = torch.randn(w.B, w.Hkv, w.T, w.d, generator=g, dtype=torch.float32).to(dt)
    v = torch.randn(w.B, w.Hkv, w.T, w.d, generator=g, dtype=torch.float32).to(dt)
    if w.qk_mult != 1.0:
        m = float(w.qk_mult)
        assert math.log2(m).is_integer(), "qk_mult must be a power of two (exact scaling)"
        q = q * m
        k = k * m
    return q.contiguous(), k.contiguous(), v.contiguous()


def make_chunk_inputs(w: ChunkWorkload, seed: Optional[int] = None):
    """Return CPU tensors q [B,Hq,Tq,d], k, v [B,Hkv,Tk,d] in the workload dtype."""
    g = _gen(w.seed if seed is None else seed)
    dt = torch_dtype(w.dtype)
    q = torch.randn(w.B, w.Hq, w.Tq, w.d, generator=g, dtype=torch.float32).to(dt)
    k = torch.randn(w.B, w.Hkv, w.Tk, w.d, generator=g, dtype=torch.float32).to(dt)
    v = torch.randn(w.B, w.Hkv, w.Tk, w.d, generator=g, dtype=torch.float32).to(dt)
    return q.contiguous(), k.contiguous(), v.contiguous()


def make_decode_inputs(w: DecodeWorkload, seed: Optional[int] = None,
                       seq_lens: Optional[torch.Tensor] = None, nan_fill: bool = True):
    """Return CPU tensors (q [B,Hq,1,d], k_cache, v_cache [B,Hkv,Lmax,d], seq_lens int32 [B])."""
    g = _gen(w.seed if seed is None else seed)
    dt = torch_dtype(w.dtype)
    drawn = torch.randint(w.Lmin, w.Lmax + 1, (w.B,), generator=g, dtype=torch.int64)
    if seq_lens is None:
        seq_lens = drawn
    seq_lens = torch.as_tensor(seq_lens, dtype=torch.int64)
    q = torch.randn(w.B, w.Hq, 1, w.d, generator=g, dtype=torch.float32).to(dt)
    fill = float("nan") if nan_fill else 0.0
    k_cache = torch.full((w.B, w.Hkv, w.Lmax, w.d), fill, dtype=dt)
    v_cache = torch.full((w.B, w.Hkv, w.Lmax, w.d), fill, dtype=dt)
    for b in range(w.B):
        L = int(seq_lens[b])
        k_cache[b, :, :L] = torch.randn(w.Hkv, L, w.d, generator=g, dtype=torch.float32).to(dt)
        v_cache[b, :, :L] = torch.randn(w.Hkv, L, w.d, generator=g, dtype=torch.float32).to(dt)
    return q.contiguous(), k_cache, v_cache, seq_lens.to(torch.int32)


def page_cache(k_cache: torch.Tensor, v_cache: torch.Tensor, seq_lens, page_size: int,
               seed: int = 0, spare: int = 0):
    """Scatter contiguous caches [B, Hkv, Lmax, d] into a shuffled pool of pages.

    Returns (k_pages, v_pages [num_pages, Hkv, page_size, d], block_table int32
    [B, ceil(Lmax / page_size)]) on the caches' device: the pages that hold rows
    < seq_lens[b] go to seeded random slots of the pool, `spare` unused pages are
    added, and table entries past a sequence's last page are -1.  Pure data
    placement: row t of sequence b ends up in page table[b, t // page_size] at
    offset t % page_size.
    """
    B, Hkv, Lmax, d = k_cache.shape
    dev = k_cache.device
    max_pages = -(-Lmax // page_size)
    pad = max_pages * page_size - Lmax
    lens = torch.as_tensor(seq_lens, dtype=torch.int64).cpu()
    used = torch.arange(max_pages).unsqueeze(0) < (-(-lens // page_size)).unsqueeze(1)
    n_used = int(used.sum())
    num_pages = n_used + spare
    perm = torch.randperm(num_pages, generator=_gen(seed))[:n_used]
    table = torch.full((B, max_pages), -1, dtype=torch.int32)
    table[used] = perm.to(torch.int32)
    sel = used.reshape(-1).nonzero().squeeze(1).to(dev)
    out = []
    for c in (k_cache, v_cache):
        if pad:
            c = torch.nn.functional.pad(c, (0, 0, 0, pad))
        blocks = c.reshape(B, Hkv, max_pages, page_size, d).permute(0, 2, 1, 3, 4)
        blocks = blocks.reshape(B * max_pages, Hkv, page_size, d)
        pool = torch.zeros(num_pages, Hkv, page_size, d, dtype=c.dtype, device=dev)
        pool[perm.to(dev)] = blocks.index_select(0, sel)
        out.append(pool)
    return out[0], out[1], table.to(dev)


def sample_query_rows(T: int, n: int, seed: int) -> list:
    """Seeded subset of query rows for sampled parity; always holds the tile edges."""
    fixed = {0, 1, 127, 128, T - 1, T // 2, min(T - 1, 255), min(T - 1, 256)}
    fixed = {r for r in fixed if 0 <= r < T}
    g = _gen(seed + 7919)
    extra = torch.randperm(T, generator=g)[: max(0, n - len(fixed))].tolist()
    return sorted(fixed.union(extra))
