"""csattn_attn_decode_noalloc: the decode entry point that allocates nothing.

Some callers cannot allocate device memory when they decode (a plugin inside a
framework that owns all device memory, a latency-critical loop where cudaMalloc
would synchronise the device).  For them the library keeps the split partials
in a static device buffer instead of a caller workspace.  These tests call the
entry point through the C ABI and hold its output to the regular
csattn_attn_decode on the same inputs: the same kernels with the same split
count, so the two must agree bit for bit.  Three calls run in a row with
different inputs, the last with much shorter sequences (fewer splits) than the
one before, so partials left in the shared buffer by an earlier call would show
if the merge read them.  The file is named to be collected last.
"""
import math

import pytest
import torch

import attn_workloads as W
import transformer_causal_self_gb300 as csattn
from tests.gpu_helpers import dev

pytestmark = pytest.mark.gpu


def _call_noalloc(lib, q, kc, vc, sl, out, w, max_len, splits):
    return lib.csattn_attn_decode_noalloc(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), sl.data_ptr(),
                                          out.data_ptr(), w.B, w.Hq, w.Hkv, w.Lmax, w.d, 1,
                                          float(w.scale), int(max_len), int(splits),
                                          torch.cuda.current_stream().cuda_stream)


def _inputs(seed, shrink=1):
    w = W.WORKLOADS["decode_bf16"].with_(B=16, Lmax=4096, Lmin=1, seed=seed)
    q, kc, vc, sl = (t.to(dev()) for t in W.make_decode_inputs(w))
    if shrink > 1:  # shorter sequences over the same cache (rows past them are not read)
        sl = torch.clamp(sl // shrink, min=1)
    return w, q, kc, vc, sl


@pytest.mark.parametrize("splits", [0, 5])
def test_noalloc_decode_matches_workspace_decode(splits):
    lib = csattn.load_library()
    for seed, shrink in ((11, 1), (12, 1), (13, 16)):  # three calls in a row, the last short
        w, q, kc, vc, sl = _inputs(seed, shrink)
        max_len = int(sl.max().item())
        ref = csattn.attn_decode(q, kc, vc, sl, scale=w.scale, max_seq_len=max_len,
                                 num_splits=splits)
        csattn.check_status()
        out = torch.full_like(q, float("nan"))
        rc = _call_noalloc(lib, q, kc, vc, sl, out, w, max_len, splits)
        assert rc == 0, lib.csattn_last_error()
        csattn.check_status()
        assert torch.equal(out, ref), f"noalloc seed {seed}: differs from the workspace decode"


def test_noalloc_second_call_reserves_no_device_memory():
    lib = csattn.load_library()
    w, q, kc, vc, sl = _inputs(14)
    max_len = int(sl.max().item())
    out = torch.empty_like(q)
    assert _call_noalloc(lib, q, kc, vc, sl, out, w, max_len, 0) == 0, lib.csattn_last_error()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    assert _call_noalloc(lib, q, kc, vc, sl, out, w, max_len, 0) == 0, lib.csattn_last_error()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    csattn.check_status()
    assert free1 == free0


def test_noalloc_rejects_partials_beyond_the_static_buffer():
    lib = csattn.load_library()
    w = W.DecodeWorkload("big", B=64, Hq=32, Hkv=8, d=128, Lmax=8192, Lmin=1,
                         scale=1.0 / math.sqrt(128))
    # 128 splits need 64*32*128*130*4 bytes of partials, far above the buffer;
    # the call must refuse before launching anything, so the tensors stay unread
    q = torch.empty(64, 32, 1, 128, dtype=torch.bfloat16, device=dev())
    kc = torch.empty(64, 8, 8192, 128, dtype=torch.bfloat16, device=dev())
    sl = torch.full((64,), 8192, dtype=torch.int32, device=dev())
    out = torch.empty_like(q)
    rc = _call_noalloc(lib, q, kc, kc, sl, out, w, 8192, 128)
    assert rc == -5
    msg = lib.csattn_last_error().decode()
    assert "static scratch" in msg and str(16 * 1024 * 1024) in msg
    csattn.check_status()
