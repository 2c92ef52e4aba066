"""Python binding of libcsattn, the sm_103a causal GQA attention library.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in include/csattn.h.  PyTorch provides the
device memory (tensors, workspaces) and the stream.  There is no CPU fallback:
if the library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

__all__ = [
    "CsattnError", "library_path", "load_library", "attn_fwd", "attn_fwd_host", "attn_fwd_ext",
    "attn_bwd", "attn_bwd_ext", "attn_decode", "attn_decode_ext", "attn_decode_host",
    "attn_decode_step",
    "attn_decode_paged", "attn_prefill_paged", "cache_append", "cache_append_paged",
    "rope_rotate", "fwd_workspace_size", "fwd_ext_workspace_size", "fwd_host_workspace_size",
    "bwd_workspace_size", "bwd_ext_workspace_size", "decode_workspace_size",
    "decode_host_workspace_size", "decode_step_workspace_size", "check_status",
    "selftest_bounded_wait", "EXPORTED_SYMBOLS",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB: Optional[ctypes.CDLL] = None

CSATTN_F32, CSATTN_BF16 = 0, 1
K_PREROTATED = 0x100
_ROPE_LAYOUT = {"split_half": 0, "adjacent": 1}
_STATUS = {0: "CSATTN_OK", -1: "CSATTN_ERR_INVALID_ARG", -2: "CSATTN_ERR_UNSUPPORTED",
           -3: "CSATTN_ERR_CUDA", -4: "CSATTN_ERR_TIMEOUT", -5: "CSATTN_ERR_WORKSPACE",
           -6: "CSATTN_ERR_DEVICE_ARG"}

_c_int, _c_float, _c_size, _vp = ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p

# name -> (restype, argtypes); the C declarations are in include/csattn.h
_SIGNATURES = {
    "csattn_fwd_workspace_size": (_c_size, [_c_int] * 6 + [_c_float]),
    "csattn_attn_fwd": (_c_int, [_vp, _vp, _vp, _vp] + [_c_int] * 7 + [_c_float, _c_int, _c_float,
                                                                        _vp, _vp, _c_size, _vp]),
    "csattn_fwd_host_workspace_size": (_c_size, [_c_int] * 6 + [_c_float]),
    "csattn_attn_fwd_host": (_c_int, [_vp] * 4 + [_c_int] * 7 + [_c_float, _c_int, _c_float, _vp,
                                                                 _c_int, _vp, _c_size, _vp]),
    "csattn_decode_host_workspace_size": (_c_size, [_c_int] * 6),
    "csattn_attn_decode_host": (_c_int, [_vp] * 5 + [_c_int] * 6 + [_c_float, _c_int, _c_int, _vp,
                                                                    _c_size, _vp]),
    "csattn_fwd_ext_workspace_size": (_c_size, [_c_int] * 7 + [_c_float]),
    "csattn_attn_fwd_ext": (_c_int, [_vp, _vp, _vp, _vp] + [_c_int] * 10 + [_c_float, _c_int,
                                                                            _c_float, _vp, _vp,
                                                                            _c_size, _vp]),
    "csattn_bwd_workspace_size": (_c_size, [_c_int] * 6 + [_c_float]),
    "csattn_attn_bwd": (_c_int, [_vp] * 9 + [_c_int] * 7 + [_c_float, _c_int, _c_float, _vp,
                                                             _c_size, _vp]),
    "csattn_bwd_ext_workspace_size": (_c_size, [_c_int] * 7 + [_c_float]),
    "csattn_attn_bwd_ext": (_c_int, [_vp] * 9 + [_c_int] * 10 + [_c_float, _c_int, _c_float, _vp,
                                                                  _c_size, _vp]),
    "csattn_rope_rotate": (_c_int, [_vp, _vp] + [_c_int] * 5 + [_c_float, _c_int, _vp]),
    "csattn_decode_workspace_size": (_c_size, [_c_int] * 5),
    "csattn_attn_decode": (_c_int, [_vp] * 5 + [_c_int] * 6 + [_c_float, _c_int, _c_int, _vp,
                                                                _c_size, _vp]),
    "csattn_attn_decode_ext": (_c_int, [_vp] * 5 + [_c_int] * 7 + [_c_float, _c_int, _c_int, _vp,
                                                                    _c_size, _vp]),
    "csattn_attn_decode_noalloc": (_c_int, [_vp] * 5 + [_c_int] * 6 + [_c_float, _c_int, _c_int,
                                                                        _vp]),
    "csattn_decode_step_workspace_size": (_c_size, [_c_int] * 5),
    "csattn_attn_decode_step": (_c_int, [_vp] * 7 + [_c_int] * 6 + [_c_float, _c_int, _c_float,
                                                                    _c_int, _c_int, _vp, _c_size,
                                                                    _vp]),
    "csattn_attn_decode_paged": (_c_int, [_vp] * 6 + [_c_int] * 8 + [_c_float, _c_int, _c_int, _vp,
                                                                    _c_size, _vp]),
    "csattn_attn_prefill_paged": (_c_int, [_vp] * 6 + [_c_int] * 10 + [_c_float, _c_int, _c_float,
                                                                     _vp, _vp, _c_size, _vp]),
    "csattn_prefill_paged_workspace_size": (_c_size, [_c_int] * 5),
    "csattn_cache_append": (_c_int, [_vp] * 5 + [_c_int] * 6 + [_c_float, _c_int, _vp]),
    "csattn_cache_append_paged": (_c_int, [_vp] * 6 + [_c_int] * 8 + [_c_float, _c_int, _vp]),
    "csattn_check_status": (_c_int, [_vp]),
    "csattn_selftest_bounded_wait": (_c_int, [_c_int, _vp]),
    "csattn_last_error": (ctypes.c_char_p, []),
    "csattn_status_str": (ctypes.c_char_p, [_c_int]),
    "csattn_version": (_c_int, []),
}
EXPORTED_SYMBOLS = tuple(_SIGNATURES)


class CsattnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_STATUS.get(status, status)}: {message}")
        self.status = status


def library_path() -> str:
    return os.path.join(_HERE, "libcsattn.so")


def load_library() -> ctypes.CDLL:
    """Load libcsattn.so (built by __graft_entry__.build()); raises if it is missing."""
    global _LIB
    if _LIB is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is not built: run `python -c 'import __graft_entry__ as g; "
                               "g.build()'` first (there is no CPU fallback)")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
    return _LIB


def _check(status: int) -> None:
    if status != 0:
        msg = load_library().csattn_last_error()
        raise CsattnError(status, msg.decode() if msg else "")


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return CSATTN_BF16
    if t.dtype == torch.float32:
        return CSATTN_F32
    raise TypeError(f"unsupported dtype {t.dtype} (bf16 or fp32)")


def _need_cuda(*ts):
    for t in ts:
        if not t.is_cuda:
            raise ValueError("tensors must be on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def fwd_workspace_size(B, Hq, Hkv, T, d, dtype: torch.dtype, rope_base: float) -> int:
    code = CSATTN_BF16 if dtype == torch.bfloat16 else CSATTN_F32
    return int(load_library().csattn_fwd_workspace_size(B, Hq, Hkv, T, d, code, float(rope_base)))


def fwd_ext_workspace_size(B, Hq, Hkv, Tq, Tk, d, dtype: torch.dtype, rope_base: float) -> int:
    code = CSATTN_BF16 if dtype == torch.bfloat16 else CSATTN_F32
    return int(load_library().csattn_fwd_ext_workspace_size(B, Hq, Hkv, Tq, Tk, d, code,
                                                            float(rope_base)))


def bwd_ext_workspace_size(B, Hq, Hkv, Tq, Tk, d, dtype: torch.dtype, rope_base: float) -> int:
    code = CSATTN_BF16 if dtype == torch.bfloat16 else CSATTN_F32
    return int(load_library().csattn_bwd_ext_workspace_size(B, Hq, Hkv, Tq, Tk, d, code,
                                                            float(rope_base)))


def bwd_workspace_size(B, Hq, Hkv, T, d, dtype: torch.dtype, rope_base: float) -> int:
    code = CSATTN_BF16 if dtype == torch.bfloat16 else CSATTN_F32
    return int(load_library().csattn_bwd_workspace_size(B, Hq, Hkv, T, d, code, float(rope_base)))


def decode_step_workspace_size(B, Hq, Lmax, d, num_splits: int = 0) -> int:
    return int(load_library().csattn_decode_step_workspace_size(B, Hq, Lmax, d, num_splits))


def decode_workspace_size(B, Hq, Lmax, d, num_splits: int = 0) -> int:
    return int(load_library().csattn_decode_workspace_size(B, Hq, Lmax, d, num_splits))


def rope_rotate(x: torch.Tensor, out: Optional[torch.Tensor] = None, *, rope_base: float,
                rope_layout: str = "split_half", stream=None) -> torch.Tensor:
    """RoPE of x [B,H,T,d] (bf16) at positions 0..T-1 (C: csattn_rope_rotate)."""
    _need_cuda(x)
    B, H, T, d = x.shape
    if out is None:
        out = torch.empty_like(x)
    _need_cuda(out)
    _check(load_library().csattn_rope_rotate(x.data_ptr(), out.data_ptr(), B, H, T, d,
                                             _dtype_code(x), float(rope_base),
                                             _ROPE_LAYOUT[rope_layout], _stream_handle(stream)))
    return out


def attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: Optional[torch.Tensor] = None,
             *, causal: bool = True, rope_base: float = 0.0, scale: float = 0.0,
             rope_layout: str = "split_half", lse: Optional[torch.Tensor] = None,
             workspace: Optional[torch.Tensor] = None, k_prerotated: bool = False,
             stream=None) -> torch.Tensor:
    """out = softmax(RoPE(q) RoPE(k)^T * scale + M) v  (C: csattn_attn_fwd).

    q [B,Hq,T,d], k/v [B,Hkv,T,d] (bf16 or fp32, contiguous, CUDA).  scale <= 0
    means 1/sqrt(d); rope_base <= 0 means no RoPE.  lse, if given, is an fp32
    [B,Hq,T] tensor that receives the natural-log log-sum-exp of each row.
    """
    _need_cuda(q, k, v)
    B, Hq, T, d = q.shape
    Hkv = k.shape[1]
    if out is None:
        out = torch.empty_like(q)
    _need_cuda(out)
    if lse is not None:
        _need_cuda(lse)
    need = 0 if k_prerotated else fwd_workspace_size(B, Hq, Hkv, T, d, q.dtype, rope_base)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    lib = load_library()
    _check(lib.csattn_attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, Hq, Hkv,
                               T, d, _dtype_code(q), int(bool(causal)), float(rope_base),
                               _ROPE_LAYOUT[rope_layout] | (K_PREROTATED if k_prerotated else 0),
                               float(scale),
                               lse.data_ptr() if lse is not None else None, ws_ptr, ws_bytes,
                               _stream_handle(stream)))
    return out


def _need_host(*ts):
    for t in ts:
        if t.device.type != "cpu":
            raise ValueError("host tensors expected")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def fwd_host_workspace_size(B, Hq, Hkv, T, d, dtype: torch.dtype, rope_base: float) -> int:
    code = CSATTN_BF16 if dtype == torch.bfloat16 else CSATTN_F32
    return int(load_library().csattn_fwd_host_workspace_size(B, Hq, Hkv, T, d, code,
                                                             float(rope_base)))


def attn_fwd_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                  out: Optional[torch.Tensor] = None, *, causal: bool = True,
                  rope_base: float = 0.0, scale: float = 0.0, rope_layout: str = "split_half",
                  lse: Optional[torch.Tensor] = None, num_chunks: int = 0,
                  workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """attn_fwd on host tensors (C: csattn_attn_fwd_host): copies in, attention and
    copies out pipelined over chunks of (sequence, KV head) pairs on the current
    device.  q, k, v, out (and lse) are CPU tensors, pinned for asynchronous copies;
    out is allocated pinned when not given.  Asynchronous on `stream`: synchronize
    before reading out.
    """
    _need_host(q, k, v)
    B, Hq, T, d = q.shape
    Hkv = k.shape[1]
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    _need_host(out)
    if lse is not None:
        _need_host(lse)
    if workspace is None:
        workspace = torch.empty(fwd_host_workspace_size(B, Hq, Hkv, T, d, q.dtype, rope_base),
                                dtype=torch.uint8, device=torch.device("cuda",
                                                                       torch.cuda.current_device()))
    lib = load_library()
    _check(lib.csattn_attn_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B,
                                    Hq, Hkv, T, d, _dtype_code(q), int(bool(causal)),
                                    float(rope_base), _ROPE_LAYOUT[rope_layout], float(scale),
                                    lse.data_ptr() if lse is not None else None, int(num_chunks),
                                    workspace.data_ptr(), workspace.numel(),
                                    _stream_handle(stream)))
    return out


def decode_host_workspace_size(B, Hq, Hkv, Lmax, d, num_splits=0) -> int:
    return int(load_library().csattn_decode_host_workspace_size(B, Hq, Hkv, Lmax, d,
                                                                int(num_splits)))


def attn_decode_host(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                     seq_lens: torch.Tensor, out: Optional[torch.Tensor] = None, *,
                     scale: float = 0.0, num_splits: int = 0, num_chunks: int = 0,
                     workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """attn_decode on host tensors (C: csattn_attn_decode_host): only the cache rows
    below seq_lens cross to the device, pipelined with the decode over chunks of
    sequences.  seq_lens is an int32 CPU tensor read during the call.  Asynchronous on
    `stream`: synchronize before reading out.
    """
    _need_host(q, k_cache, v_cache, seq_lens)
    if seq_lens.dtype != torch.int32:
        raise TypeError("seq_lens must be int32")
    B, Hq, _, d = q.shape
    Hkv, Lmax = k_cache.shape[1], k_cache.shape[2]
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    _need_host(out)
    if workspace is None:
        workspace = torch.empty(decode_host_workspace_size(B, Hq, Hkv, Lmax, d, num_splits),
                                dtype=torch.uint8,
                                device=torch.device("cuda", torch.cuda.current_device()))
    lib = load_library()
    _check(lib.csattn_attn_decode_host(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                       seq_lens.data_ptr(), out.data_ptr(), B, Hq, Hkv, Lmax, d,
                                       _dtype_code(q), float(scale), int(num_splits),
                                       int(num_chunks), workspace.data_ptr(), workspace.numel(),
                                       _stream_handle(stream)))
    return out


def attn_fwd_ext(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                 out: Optional[torch.Tensor] = None, *, q_offset: int = 0, causal: bool = True,
                 rope_base: float = 0.0, scale: float = 0.0, rope_layout: str = "split_half",
                 lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                 k_prerotated: bool = False, stream=None) -> torch.Tensor:
    """Chunked / rectangular prefill (C: csattn_attn_fwd_ext).

    q [B,Hq,Tq,d], k [B,Hkv,Tk,d], v [B,Hkv,Tk,dv]; out [B,Hq,Tq,dv].  Query row i
    sits at position q_offset + i; with causal it sees keys j <= q_offset + i.  RoPE
    rotates q at q_offset + i and k at 0..Tk-1 (unless k_prerotated).  lse, if given,
    is fp32 [B,Hq,Tq].
    """
    _need_cuda(q, k, v)
    B, Hq, Tq, d = q.shape
    Hkv, Tk = k.shape[1], k.shape[2]
    dv = v.shape[3]
    if out is None:
        out = q.new_empty((B, Hq, Tq, dv))
    _need_cuda(out)
    if lse is not None:
        _need_cuda(lse)
    need = 0 if k_prerotated else fwd_ext_workspace_size(B, Hq, Hkv, Tq, Tk, d, q.dtype, rope_base)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    lib = load_library()
    _check(lib.csattn_attn_fwd_ext(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, Hq,
                                   Hkv, Tq, Tk, int(q_offset), d, dv, _dtype_code(q),
                                   int(bool(causal)), float(rope_base),
                                   _ROPE_LAYOUT[rope_layout] | (K_PREROTATED if k_prerotated else 0),
                                   float(scale), lse.data_ptr() if lse is not None else None,
                                   ws_ptr, ws_bytes, _stream_handle(stream)))
    return out


def attn_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor,
             dout: torch.Tensor, lse: torch.Tensor, *, causal: bool = True,
             rope_base: float = 0.0, scale: float = 0.0, rope_layout: str = "split_half",
             dq: Optional[torch.Tensor] = None, dk: Optional[torch.Tensor] = None,
             dv: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
             stream=None):
    """Gradients (dq, dk, dv) of sum(out * dout) (C: csattn_attn_bwd).

    out and lse are the forward's outputs for the same arguments (lse fp32 [B,Hq,T]).
    """
    _need_cuda(q, k, v, out, dout, lse)
    B, Hq, T, d = q.shape
    Hkv = k.shape[1]
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if workspace is None:
        n = bwd_workspace_size(B, Hq, Hkv, T, d, q.dtype, rope_base)
        workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=q.device)
    lib = load_library()
    _check(lib.csattn_attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                               dout.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                               dv.data_ptr(), B, Hq, Hkv, T, d, _dtype_code(q), int(bool(causal)),
                               float(rope_base), _ROPE_LAYOUT[rope_layout], float(scale),
                               workspace.data_ptr(), workspace.numel(), _stream_handle(stream)))
    return dq, dk, dv


def attn_bwd_ext(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor,
                 dout: torch.Tensor, lse: torch.Tensor, *, q_offset: int = 0, causal: bool = True,
                 rope_base: float = 0.0, scale: float = 0.0, rope_layout: str = "split_half",
                 dq: Optional[torch.Tensor] = None, dk: Optional[torch.Tensor] = None,
                 dv: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                 stream=None):
    """Gradients of sum(out * dout) for attn_fwd_ext (C: csattn_attn_bwd_ext).

    q [B,Hq,Tq,d], k [B,Hkv,Tk,d], v [B,Hkv,Tk,dv]; out, dout [B,Hq,Tq,dv]; lse fp32
    [B,Hq,Tq] from the forward with the same q_offset, causal and RoPE arguments.
    Returns dq, dk, dv shaped like q, k, v.
    """
    _need_cuda(q, k, v, out, dout, lse)
    B, Hq, Tq, d = q.shape
    Hkv, Tk = k.shape[1], k.shape[2]
    d_v = v.shape[3]
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _need_cuda(dq, dk, dv)
    if workspace is None:
        n = bwd_ext_workspace_size(B, Hq, Hkv, Tq, Tk, d, q.dtype, rope_base)
        workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=q.device)
    lib = load_library()
    _check(lib.csattn_attn_bwd_ext(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                   dout.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                   dv.data_ptr(), B, Hq, Hkv, Tq, Tk, int(q_offset), d, d_v,
                                   _dtype_code(q), int(bool(causal)), float(rope_base),
                                   _ROPE_LAYOUT[rope_layout], float(scale), workspace.data_ptr(),
                                   workspace.numel(), _stream_handle(stream)))
    return dq, dk, dv


def attn_decode_ext(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                    seq_lens: torch.Tensor, out: Optional[torch.Tensor] = None, *,
                    scale: float = 0.0, max_seq_len: Optional[int] = None, num_splits: int = 0,
                    workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """KV-cache decode with a value width of its own (C: csattn_attn_decode_ext).

    q [B,Hq,1,d], k_cache [B,Hkv,Lmax,d], v_cache [B,Hkv,Lmax,dv]; returns out
    [B,Hq,1,dv].  Otherwise as attn_decode.
    """
    _need_cuda(q, k_cache, v_cache, seq_lens)
    if seq_lens.dtype != torch.int32:
        raise TypeError("seq_lens must be int32")
    B, Hq, _, d = q.shape
    Hkv, Lmax, dv = k_cache.shape[1], k_cache.shape[2], v_cache.shape[3]
    if max_seq_len is None:
        max_seq_len = Lmax
    if out is None:
        out = q.new_empty((B, Hq, 1, dv))
    _need_cuda(out)
    if workspace is None:
        workspace = torch.empty(decode_workspace_size(B, Hq, Lmax, dv, num_splits),
                                dtype=torch.uint8, device=q.device)
    lib = load_library()
    _check(lib.csattn_attn_decode_ext(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                      seq_lens.data_ptr(), out.data_ptr(), B, Hq, Hkv, Lmax, d,
                                      dv, _dtype_code(q), float(scale), int(max_seq_len),
                                      int(num_splits), workspace.data_ptr(), workspace.numel(),
                                      _stream_handle(stream)))
    return out


def attn_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                seq_lens: torch.Tensor, out: Optional[torch.Tensor] = None, *, scale: float = 0.0,
                max_seq_len: Optional[int] = None, num_splits: int = 0,
                workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """KV-cache decode (C: csattn_attn_decode).

    q [B,Hq,1,d] already rotated; k_cache/v_cache [B,Hkv,Lmax,d]; seq_lens int32
    [B] on the device.  max_seq_len defaults to Lmax (always a valid bound).
    """
    _need_cuda(q, k_cache, v_cache, seq_lens)
    if seq_lens.dtype != torch.int32:
        raise TypeError("seq_lens must be int32")
    B, Hq, _, d = q.shape
    Hkv, Lmax = k_cache.shape[1], k_cache.shape[2]
    if max_seq_len is None:
        max_seq_len = Lmax
    if out is None:
        out = torch.empty_like(q)
    _need_cuda(out)
    if workspace is None:
        workspace = torch.empty(decode_workspace_size(B, Hq, Lmax, d, num_splits),
                                dtype=torch.uint8, device=q.device)
    lib = load_library()
    _check(lib.csattn_attn_decode(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                  seq_lens.data_ptr(), out.data_ptr(), B, Hq, Hkv, Lmax, d,
                                  _dtype_code(q), float(scale), int(max_seq_len), int(num_splits),
                                  workspace.data_ptr(), workspace.numel(), _stream_handle(stream)))
    return out


def attn_decode_step(q_new: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                     k_cache: torch.Tensor, v_cache: torch.Tensor, cache_lens: torch.Tensor,
                     out: Optional[torch.Tensor] = None, *, rope_base: float = 0.0,
                     rope_layout: str = "split_half", scale: float = 0.0,
                     max_seq_len: Optional[int] = None, num_splits: int = 0,
                     workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Decode step with the cache append fused in (C: csattn_attn_decode_step).

    q_new [B,Hq,1,d], k_new/v_new [B,Hkv,1,d] not rotated; the caches are written at
    row cache_lens[b] (int32 [B] on the device, not modified); the query attends to
    rows 0..cache_lens[b].  max_seq_len bounds cache_lens + 1 (default Lmax).
    """
    _need_cuda(q_new, k_new, v_new, k_cache, v_cache, cache_lens)
    if cache_lens.dtype != torch.int32:
        raise TypeError("cache_lens must be int32")
    B, Hq, _, d = q_new.shape
    Hkv, Lmax = k_cache.shape[1], k_cache.shape[2]
    if max_seq_len is None:
        max_seq_len = Lmax
    if out is None:
        out = torch.empty_like(q_new)
    _need_cuda(out)
    if workspace is None:
        workspace = torch.empty(decode_step_workspace_size(B, Hq, Lmax, d, num_splits),
                                dtype=torch.uint8, device=q_new.device)
    lib = load_library()
    _check(lib.csattn_attn_decode_step(q_new.data_ptr(), k_new.data_ptr(), v_new.data_ptr(),
                                       k_cache.data_ptr(), v_cache.data_ptr(),
                                       cache_lens.data_ptr(), out.data_ptr(), B, Hq, Hkv, Lmax, d,
                                       _dtype_code(q_new), float(rope_base),
                                       _ROPE_LAYOUT[rope_layout], float(scale), int(max_seq_len),
                                       int(num_splits), workspace.data_ptr(), workspace.numel(),
                                       _stream_handle(stream)))
    return out


def attn_decode_paged(q: torch.Tensor, k_pages: torch.Tensor, v_pages: torch.Tensor,
                      block_table: torch.Tensor, seq_lens: torch.Tensor,
                      out: Optional[torch.Tensor] = None, *, scale: float = 0.0,
                      max_seq_len: Optional[int] = None, num_splits: int = 0,
                      workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Decode over a paged cache (C: csattn_attn_decode_paged).

    k_pages/v_pages [num_pages, Hkv, page_size, d]; block_table int32 [B, max_pages] and
    seq_lens int32 [B] on the device.  max_seq_len defaults to max_pages * page_size.
    """
    _need_cuda(q, k_pages, v_pages, block_table, seq_lens)
    if block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("block_table and seq_lens must be int32")
    B, Hq, _, d = q.shape
    num_pages, Hkv, page_size = k_pages.shape[0], k_pages.shape[1], k_pages.shape[2]
    max_pages = block_table.shape[1]
    if max_seq_len is None:
        max_seq_len = max_pages * page_size
    if out is None:
        out = torch.empty_like(q)
    _need_cuda(out)
    if workspace is None:
        workspace = torch.empty(decode_workspace_size(B, Hq, max_pages * page_size, d, num_splits),
                                dtype=torch.uint8, device=q.device)
    lib = load_library()
    _check(lib.csattn_attn_decode_paged(q.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(),
                                        block_table.data_ptr(), seq_lens.data_ptr(), out.data_ptr(),
                                        B, Hq, Hkv, page_size, num_pages, max_pages, d,
                                        _dtype_code(q), float(scale), int(max_seq_len),
                                        int(num_splits), workspace.data_ptr(), workspace.numel(),
                                        _stream_handle(stream)))
    return out


def attn_prefill_paged(q: torch.Tensor, k_pages: torch.Tensor, v_pages: torch.Tensor,
                       block_table: torch.Tensor, cache_lens: torch.Tensor,
                       out: Optional[torch.Tensor] = None, *, causal: bool = True,
                       rope_base: float = 0.0, scale: float = 0.0,
                       rope_layout: str = "split_half", lse: Optional[torch.Tensor] = None,
                       workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Chunk prefill over a paged cache (C: csattn_attn_prefill_paged).

    q [B,Hq,Tq,d] (not rotated; row i of sequence b sits at cache_lens[b] + i);
    k_pages/v_pages [num_pages,Hkv,page_size,d] holding rotated keys, the chunk's own
    rows included; block_table int32 [B,max_pages] and cache_lens int32 [B] on the device.
    """
    _need_cuda(q, k_pages, v_pages, block_table, cache_lens)
    if block_table.dtype != torch.int32 or cache_lens.dtype != torch.int32:
        raise TypeError("block_table and cache_lens must be int32")
    B, Hq, Tq, d = q.shape
    num_pages, Hkv, page_size = k_pages.shape[0], k_pages.shape[1], k_pages.shape[2]
    max_pages = block_table.shape[1]
    if out is None:
        out = torch.empty_like(q)
    _need_cuda(out)
    lib = load_library()
    need = int(lib.csattn_prefill_paged_workspace_size(B, Hkv, page_size, max_pages, d))
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check(lib.csattn_attn_prefill_paged(q.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(),
                                         block_table.data_ptr(), cache_lens.data_ptr(),
                                         out.data_ptr(), B, Hq, Hkv, Tq, page_size, num_pages,
                                         max_pages, d, _dtype_code(q), int(bool(causal)),
                                         float(rope_base), _ROPE_LAYOUT[rope_layout],
                                         float(scale), lse.data_ptr() if lse is not None else None,
                                         workspace.data_ptr() if workspace is not None else None,
                                         workspace.numel() if workspace is not None else 0,
                                         _stream_handle(stream)))
    return out


def cache_append(k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
                 v_cache: torch.Tensor, cache_lens: torch.Tensor, *, rope_base: float = 0.0,
                 rope_layout: str = "split_half", stream=None) -> None:
    """Append Tn tokens per sequence at rows cache_lens[b].. (C: csattn_cache_append).

    k_new, v_new [B,Hkv,Tn,d] (keys not rotated); caches [B,Hkv,Lmax,d]; cache_lens
    int32 [B] on the device, not advanced.
    """
    _need_cuda(k_new, v_new, k_cache, v_cache, cache_lens)
    if cache_lens.dtype != torch.int32:
        raise TypeError("cache_lens must be int32")
    B, Hkv, Tn, d = k_new.shape
    lib = load_library()
    _check(lib.csattn_cache_append(k_new.data_ptr(), v_new.data_ptr(), k_cache.data_ptr(),
                                   v_cache.data_ptr(), cache_lens.data_ptr(), B, Hkv, Tn,
                                   k_cache.shape[2], d, _dtype_code(k_new), float(rope_base),
                                   _ROPE_LAYOUT[rope_layout], _stream_handle(stream)))


def cache_append_paged(k_new: torch.Tensor, v_new: torch.Tensor, k_pages: torch.Tensor,
                       v_pages: torch.Tensor, block_table: torch.Tensor, cache_lens: torch.Tensor,
                       *, rope_base: float = 0.0, rope_layout: str = "split_half",
                       stream=None) -> None:
    """Append into paged caches [num_pages,Hkv,page_size,d] (C: csattn_cache_append_paged)."""
    _need_cuda(k_new, v_new, k_pages, v_pages, block_table, cache_lens)
    if block_table.dtype != torch.int32 or cache_lens.dtype != torch.int32:
        raise TypeError("block_table and cache_lens must be int32")
    B, Hkv, Tn, d = k_new.shape
    num_pages, page_size = k_pages.shape[0], k_pages.shape[2]
    lib = load_library()
    _check(lib.csattn_cache_append_paged(k_new.data_ptr(), v_new.data_ptr(), k_pages.data_ptr(),
                                         v_pages.data_ptr(), block_table.data_ptr(),
                                         cache_lens.data_ptr(), B, Hkv, Tn, page_size, num_pages,
                                         block_table.shape[1], d, _dtype_code(k_new),
                                         float(rope_base), _ROPE_LAYOUT[rope_layout],
                                         _stream_handle(stream)))


def check_status(stream=None) -> None:
    """Synchronize the stream and raise if a kernel reported a timeout or a device-side error."""
    _check(load_library().csattn_check_status(_stream_handle(stream)))


def selftest_bounded_wait(limit_us: int, stream=None) -> None:
    """Launch the kernel whose barrier wait must run out (see csattn_selftest_bounded_wait)."""
    _check(load_library().csattn_selftest_bounded_wait(int(limit_us), _stream_handle(stream)))
