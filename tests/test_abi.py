"""The C-ABI library loads, exports every symbol include/csattn.h declares, and
rejects invalid arguments on the host.  No GPU needed: no call here reaches a
kernel launch or any CUDA runtime call."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "csattn.h")


def declared_symbols():
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(csattn_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    import transformer_causal_self_gb300 as csattn
    return csattn.load_library()


def test_header_declares_entry_points():
    names = declared_symbols()
    for must in ("csattn_attn_fwd", "csattn_attn_decode", "csattn_fwd_workspace_size",
                 "csattn_decode_workspace_size", "csattn_check_status", "csattn_last_error",
                 "csattn_status_str"):
        assert must in names


def test_binding_covers_header():
    import transformer_causal_self_gb300 as csattn
    assert sorted(csattn.EXPORTED_SYMBOLS) == declared_symbols()


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert getattr(lib, name) is not None
    out = subprocess.run(["nm", "-D", "--defined-only", lib._name], capture_output=True, text=True)
    assert out.returncode == 0
    exported = set(line.split()[-1] for line in out.stdout.splitlines() if " T " in line)
    missing = [n for n in declared_symbols() if n not in exported]
    assert not missing, missing


def test_status_strings_and_version(lib):
    assert lib.csattn_status_str(0) == b"CSATTN_OK"
    assert lib.csattn_status_str(-4) == b"CSATTN_ERR_TIMEOUT"
    assert lib.csattn_status_str(123) == b"CSATTN_UNKNOWN_STATUS"
    assert lib.csattn_version() >= 100


def test_workspace_sizes(lib):
    # rotated keys B*Hkv*T*d bf16 for bf16 + RoPE; nothing otherwise
    assert lib.csattn_fwd_workspace_size(4, 32, 8, 4096, 128, 1, 10000.0) == 4 * 8 * 4096 * 128 * 2
    assert lib.csattn_fwd_workspace_size(4, 32, 8, 4096, 128, 1, 0.0) == 0
    assert lib.csattn_fwd_workspace_size(1, 2, 2, 64, 16, 0, 10000.0) == 0
    # decode partials: B*Hq*splits*(d+2) fp32, automatic splits cover Lmax/256
    assert lib.csattn_fwd_ext_workspace_size(4, 32, 8, 1024, 4096, 128, 1, 10000.0) == 4 * 8 * 4096 * 128 * 2
    assert lib.csattn_fwd_ext_workspace_size(4, 32, 8, 1024, 4096, 128, 0, 10000.0) == 0
    assert lib.csattn_decode_workspace_size(64, 32, 8192, 128, 0) == 64 * 32 * 32 * 130 * 4
    assert lib.csattn_decode_workspace_size(2, 4, 100, 64, 5) == 2 * 4 * 5 * 66 * 4
    # decode step: partials rounded up to 256 bytes, then the rotated queries
    part = 2 * 4 * 5 * 66 * 4
    assert lib.csattn_decode_step_workspace_size(2, 4, 100, 64, 5) == ((part + 255) // 256) * 256 + 2 * 4 * 64 * 2


FAKE = 0x10000  # 16-byte aligned, never dereferenced: every case below fails before any CUDA call


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), -1),
    (dict(B=0), -1),
    (dict(T=0), -1),
    (dict(Hq=6, Hkv=4), -1),
    (dict(dtype=7), -1),
    (dict(causal=2), -1),
    (dict(rope_layout=5), -1),
    (dict(scale=float("nan")), -1),
    (dict(d=48), -2),
    (dict(dtype=1, d=16), -2),
    (dict(dtype=1, d=32), -2),
    (dict(T=1 << 24), -2),
    (dict(T=60000, rope_base=10000.0), -2),
    (dict(q=FAKE + 8), -1),
    (dict(lse=FAKE + 2), -1),
    (dict(dtype=1, rope_base=10000.0, ws=None, ws_bytes=0), -5),
    (dict(dtype=1, rope_base=10000.0, ws=FAKE, ws_bytes=100), -5),
])
def test_fwd_rejects_invalid_arguments(lib, kw, status):
    a = dict(q=FAKE, k=FAKE, v=FAKE, out=FAKE, B=1, Hq=4, Hkv=2, T=64, d=64, dtype=0, causal=1,
             rope_base=0.0, rope_layout=0, scale=0.0, lse=None, ws=None, ws_bytes=0)
    a.update(kw)
    rc = lib.csattn_attn_fwd(a["q"], a["k"], a["v"], a["out"], a["B"], a["Hq"], a["Hkv"], a["T"],
                             a["d"], a["dtype"], a["causal"], a["rope_base"], a["rope_layout"],
                             a["scale"], a["lse"], a["ws"], a["ws_bytes"], None)
    assert rc == status, lib.csattn_last_error()
    assert len(lib.csattn_last_error()) > 0


@pytest.mark.parametrize("kw,status", [
    (dict(q_offset=-1), -1),
    (dict(Tk=0), -1),
    (dict(Tq=0), -1),
    (dict(q_offset=1 << 24), -2),
    (dict(dtype=1, rope_base=10000.0, q_offset=49000, Tq=200), -2),
    (dict(dtype=1, rope_base=10000.0, Tk=50000), -2),
    (dict(dtype=1, rope_base=10000.0, ws=None, ws_bytes=0), -5),
    (dict(dtype=1, rope_base=10000.0, Tk=512, ws=FAKE, ws_bytes=1 * 2 * 256 * 64 * 2), -5),
    (dict(dv=96), -2),
    (dict(dtype=1, dv=32), -2),
    (dict(dtype=1, d=32, dv=64), -2),
])
def test_fwd_ext_rejects_invalid_arguments(lib, kw, status):
    a = dict(q=FAKE, k=FAKE, v=FAKE, out=FAKE, B=1, Hq=4, Hkv=2, Tq=64, Tk=256, q_offset=192,
             d=64, dv=0, dtype=0, causal=1, rope_base=0.0, rope_layout=0, scale=0.0, lse=None,
             ws=None, ws_bytes=0)
    a.update(kw)
    rc = lib.csattn_attn_fwd_ext(a["q"], a["k"], a["v"], a["out"], a["B"], a["Hq"], a["Hkv"],
                                 a["Tq"], a["Tk"], a["q_offset"], a["d"], a["dv"], a["dtype"],
                                 a["causal"],
                                 a["rope_base"], a["rope_layout"], a["scale"], a["lse"], a["ws"],
                                 a["ws_bytes"], None)
    assert rc == status, lib.csattn_last_error()
    assert b"attn_fwd_ext" in lib.csattn_last_error()


@pytest.mark.parametrize("kw,status", [
    (dict(seq=None), -1),
    (dict(B=0), -1),
    (dict(Hq=6, Hkv=4), -1),
    (dict(dtype=0, d=48), -2),
    (dict(dtype=0, d=256), -2),
    (dict(dtype=0, Hq=6, Hkv=4), -1),
    (dict(dtype=0, splits=2, ws=FAKE, ws_bytes=16), -5),
    (dict(dtype=9), -1),
    (dict(d=96), -2),
    (dict(Hq=34, Hkv=2), -2),
    (dict(max_len=0), -1),
    (dict(max_len=300), -1),
    (dict(splits=-1), -1),
    (dict(out=FAKE + 4), -1),
    (dict(splits=2, ws=None, ws_bytes=0), -5),
    (dict(splits=2, ws=FAKE, ws_bytes=16), -5),
])
def test_decode_rejects_invalid_arguments(lib, kw, status):
    a = dict(q=FAKE, k=FAKE, v=FAKE, seq=FAKE, out=FAKE, B=2, Hq=8, Hkv=2, Lmax=256, d=128,
             dtype=1, scale=0.0, max_len=256, splits=0, ws=FAKE, ws_bytes=1 << 20)
    a.update(kw)
    rc = lib.csattn_attn_decode(a["q"], a["k"], a["v"], a["seq"], a["out"], a["B"], a["Hq"],
                                a["Hkv"], a["Lmax"], a["d"], a["dtype"], a["scale"], a["max_len"],
                                a["splits"], a["ws"], a["ws_bytes"], None)
    assert rc == status, lib.csattn_last_error()


@pytest.mark.parametrize("kw,status", [
    (dict(seq=None), -1),
    (dict(q=None), -1),
    (dict(B=0), -1),
    (dict(dtype=0), -2),
    (dict(dtype=9), -1),
    (dict(d=96), -2),
    (dict(max_len=300), -1),
    (dict(splits=-1), -1),
    (dict(out=FAKE + 4), -1),
    # 128 explicit splits of B=64, Hq=32, d=128 partials: 136 MB > the 16 MiB buffer
    (dict(B=64, Hq=32, Hkv=8, Lmax=8192, max_len=8192, splits=128), -5),
])
def test_decode_noalloc_rejects_invalid_arguments(lib, kw, status):
    """Every rejection happens before any CUDA call (no GPU here)."""
    a = dict(q=FAKE, k=FAKE, v=FAKE, seq=FAKE, out=FAKE, B=2, Hq=8, Hkv=2, Lmax=256, d=128,
             dtype=1, scale=0.0, max_len=256, splits=0)
    a.update(kw)
    rc = lib.csattn_attn_decode_noalloc(a["q"], a["k"], a["v"], a["seq"], a["out"], a["B"],
                                        a["Hq"], a["Hkv"], a["Lmax"], a["d"], a["dtype"],
                                        a["scale"], a["max_len"], a["splits"], None)
    assert rc == status, lib.csattn_last_error()
    msg = lib.csattn_last_error()
    assert b"attn_decode_noalloc" in msg
    if status == -5:
        assert b"static scratch" in msg and str(16 * 1024 * 1024).encode() in msg


@pytest.mark.parametrize("kw,status", [
    (dict(table=None), -1),
    (dict(table=FAKE + 2), -1),
    (dict(page_size=0), -1),
    (dict(page_size=96), -1),
    (dict(page_size=24), -1),
    (dict(num_pages=0), -1),
    (dict(max_pages=0), -1),
    (dict(max_len=4 * 128 + 1), -1),
    (dict(d=96), -2),
    (dict(dtype=0), -2),
    (dict(seq=None), -1),
    (dict(splits=2, ws=FAKE, ws_bytes=64), -5),
])
def test_decode_paged_rejects_invalid_arguments(lib, kw, status):
    a = dict(q=FAKE, k=FAKE, v=FAKE, table=FAKE, seq=FAKE, out=FAKE, B=2, Hq=8, Hkv=2,
             page_size=128, num_pages=16, max_pages=4, d=128, dtype=1, scale=0.0, max_len=512,
             splits=0, ws=FAKE, ws_bytes=1 << 24)
    a.update(kw)
    rc = lib.csattn_attn_decode_paged(a["q"], a["k"], a["v"], a["table"], a["seq"], a["out"],
                                      a["B"], a["Hq"], a["Hkv"], a["page_size"], a["num_pages"],
                                      a["max_pages"], a["d"], a["dtype"], a["scale"], a["max_len"],
                                      a["splits"], a["ws"], a["ws_bytes"], None)
    assert rc == status, lib.csattn_last_error()
    assert b"attn_decode_paged" in lib.csattn_last_error()


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), -1),
    (dict(out=None), -1),
    (dict(B=0), -1),
    (dict(Hq=6, Hkv=4), -1),
    (dict(dtype=7), -1),
    (dict(chunks=-1), -1),
    (dict(chunks=17), -1),
    (dict(ws=None), -5),
    (dict(ws_bytes=1024), -5),
    (dict(ws=FAKE + 8), -5),
    (dict(d=48), -2),
    (dict(d=32), -2),
    (dict(causal=3), -1),
    (dict(rope_layout=5), -1),
    (dict(rope_base=10000.0, T=50000), -2),
])
def test_fwd_host_rejects_invalid_arguments(lib, kw, status):
    a = dict(q=FAKE, k=FAKE, v=FAKE, out=FAKE, B=2, Hq=8, Hkv=2, T=256, d=128, dtype=1, causal=1,
             rope_base=0.0, rope_layout=0, scale=0.0, lse=None, chunks=0, ws=FAKE,
             ws_bytes=1 << 40)
    a.update(kw)
    rc = lib.csattn_attn_fwd_host(a["q"], a["k"], a["v"], a["out"], a["B"], a["Hq"], a["Hkv"],
                                  a["T"], a["d"], a["dtype"], a["causal"], a["rope_base"],
                                  a["rope_layout"], a["scale"], a["lse"], a["chunks"], a["ws"],
                                  a["ws_bytes"], None)
    assert rc == status, lib.csattn_last_error()
    assert b"attn_fwd_host" in lib.csattn_last_error()


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), -1),
    (dict(lens=None), -1),
    (dict(B=0), -1),
    (dict(lens_v=(0, 5)), -1),
    (dict(lens_v=(5, 300)), -1),
    (dict(chunks=17), -1),
    (dict(Hq=6, Hkv=4), -1),
    (dict(dtype=0), -2),
    (dict(d=96), -2),
    (dict(Hq=34, Hkv=2), -2),
    (dict(splits=-1), -1),
    (dict(ws=None), -5),
    (dict(ws_bytes=100), -5),
])
def test_decode_host_rejects_invalid_arguments(lib, kw, status):
    import ctypes
    a = dict(q=FAKE, k=FAKE, v=FAKE, out=FAKE, B=2, Hq=8, Hkv=2, Lmax=256, d=128, dtype=1,
             scale=0.0, splits=0, chunks=0, ws=FAKE, ws_bytes=1 << 40, lens_v=(5, 256))
    a.update(kw)
    lens = (ctypes.c_int32 * len(a["lens_v"]))(*a["lens_v"])
    if "lens" in kw:
        lens = None
    rc = lib.csattn_attn_decode_host(a["q"], a["k"], a["v"], lens, a["out"], a["B"], a["Hq"],
                                     a["Hkv"], a["Lmax"], a["d"], a["dtype"], a["scale"],
                                     a["splits"], a["chunks"], a["ws"], a["ws_bytes"], None)
    assert rc == status, lib.csattn_last_error()
    assert b"attn_decode_host" in lib.csattn_last_error()


def test_decode_host_workspace_size(lib):
    al = lambda x: (x + 255) // 256 * 256  # noqa: E731
    q, c = 64 * 32 * 128 * 2, 64 * 8 * 8192 * 128 * 2
    part = lib.csattn_decode_workspace_size(64, 32, 8192, 128, 0)
    assert lib.csattn_decode_host_workspace_size(64, 32, 8, 8192, 128, 0) == \
        2 * al(q) + 2 * al(c) + al(64 * 4) + al(part)
    assert lib.csattn_decode_host_workspace_size(0, 32, 8, 8192, 128, 0) == 0


def test_fwd_host_workspace_size(lib):
    al = lambda x: (x + 255) // 256 * 256  # noqa: E731
    q, k = 4 * 32 * 4096 * 128 * 2, 4 * 8 * 4096 * 128 * 2
    lse = 4 * 32 * 4096 * 4
    assert lib.csattn_fwd_host_workspace_size(4, 32, 8, 4096, 128, 1, 0.0) == \
        2 * al(q) + 2 * al(k) + al(lse)
    assert lib.csattn_fwd_host_workspace_size(4, 32, 8, 4096, 128, 1, 10000.0) == \
        2 * al(q) + 3 * al(k) + al(lse)
    assert lib.csattn_fwd_host_workspace_size(4, 32, 8, 4096, 128, 0, 10000.0) == \
        2 * al(2 * q) + 2 * al(2 * k) + al(lse)
    assert lib.csattn_fwd_host_workspace_size(4, 32, 8, 4096, 128, 5, 0.0) == 0
    assert lib.csattn_fwd_host_workspace_size(0, 32, 8, 4096, 128, 1, 0.0) == 0


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), -1),
    (dict(table=None), -1),
    (dict(lens=None), -1),
    (dict(Tq=0), -1),
    (dict(Hq=6, Hkv=4), -1),
    (dict(dtype=0), -2),
    (dict(dtype=4), -1),
    (dict(d=32), -2),
    (dict(causal=2), -1),
    (dict(rope_layout=0x100), -1),
    (dict(page_size=96), -1),
    (dict(page_size=48), -1),
    (dict(page_size=8), -1),
    (dict(num_pages=0), -1),
    (dict(max_pages=0), -1),
    (dict(Tq=600, max_pages=4, page_size=128), -1),
    (dict(max_pages=1 << 17, page_size=128), -2),
    (dict(rope_base=10000.0, max_pages=400, page_size=128), -2),
    (dict(lens=FAKE + 2), -1),
    (dict(lse=FAKE + 2), -1),
    (dict(out=FAKE + 8), -1),
    (dict(B=70000, Hq=2, Hkv=2), -2),
    (dict(page_size=16, max_pages=32), -5),
    (dict(page_size=32, max_pages=16, ws=FAKE, ws_bytes=1024), -5),
])
def test_prefill_paged_rejects_invalid_arguments(lib, kw, status):
    a = dict(q=FAKE, k=FAKE, v=FAKE, table=FAKE, lens=FAKE, out=FAKE, B=2, Hq=8, Hkv=2, Tq=256,
             page_size=128, num_pages=16, max_pages=4, d=128, dtype=1, causal=1, rope_base=0.0,
             rope_layout=0, scale=0.0, lse=None, ws=None, ws_bytes=0)
    a.update(kw)
    rc = lib.csattn_attn_prefill_paged(a["q"], a["k"], a["v"], a["table"], a["lens"], a["out"],
                                       a["B"], a["Hq"], a["Hkv"], a["Tq"], a["page_size"],
                                       a["num_pages"], a["max_pages"], a["d"], a["dtype"],
                                       a["causal"], a["rope_base"], a["rope_layout"], a["scale"],
                                       a["lse"], a["ws"], a["ws_bytes"], None)
    assert rc == status, lib.csattn_last_error()
    assert b"attn_prefill_paged" in lib.csattn_last_error()


@pytest.mark.parametrize("kw,status", [
    (dict(k_new=None), -1),
    (dict(lens=FAKE + 2), -1),
    (dict(Tn=0), -1),
    (dict(Tn=300, Lmax=256), -1),
    (dict(d=96), -2),
    (dict(dtype=0), -2),
    (dict(dtype=5), -1),
    (dict(rope_layout=3), -1),
    (dict(rope_base=10000.0, Lmax=60000, Tn=16), -2),
])
def test_cache_append_rejects_invalid_arguments(lib, kw, status):
    a = dict(k_new=FAKE, v_new=FAKE, kc=FAKE, vc=FAKE, lens=FAKE, B=2, Hkv=2, Tn=16, Lmax=256,
             d=128, dtype=1, rope_base=0.0, rope_layout=0)
    a.update(kw)
    rc = lib.csattn_cache_append(a["k_new"], a["v_new"], a["kc"], a["vc"], a["lens"], a["B"],
                                 a["Hkv"], a["Tn"], a["Lmax"], a["d"], a["dtype"], a["rope_base"],
                                 a["rope_layout"], None)
    assert rc == status, lib.csattn_last_error()
    assert b"cache_append" in lib.csattn_last_error()


@pytest.mark.parametrize("kw,status", [
    (dict(table=None), -1),
    (dict(page_size=96), -1),
    (dict(page_size=20), -1),
    (dict(num_pages=0), -1),
    (dict(Tn=600), -1),
    (dict(d=32), -2),
])
def test_cache_append_paged_rejects_invalid_arguments(lib, kw, status):
    a = dict(k_new=FAKE, v_new=FAKE, kp=FAKE, vp=FAKE, table=FAKE, lens=FAKE, B=2, Hkv=2, Tn=16,
             page_size=128, num_pages=8, max_pages=4, d=128, dtype=1, rope_base=0.0,
             rope_layout=0)
    a.update(kw)
    rc = lib.csattn_cache_append_paged(a["k_new"], a["v_new"], a["kp"], a["vp"], a["table"],
                                       a["lens"], a["B"], a["Hkv"], a["Tn"], a["page_size"],
                                       a["num_pages"], a["max_pages"], a["d"], a["dtype"],
                                       a["rope_base"], a["rope_layout"], None)
    assert rc == status, lib.csattn_last_error()
    assert b"cache_append_paged" in lib.csattn_last_error()


@pytest.mark.parametrize("kw,status", [
    (dict(q_new=None), -1),
    (dict(k_new=FAKE + 8), -1),
    (dict(rope_layout=7), -1),
    (dict(rope_base=float("inf")), -1),
    (dict(max_seq_len=0), -1),
    (dict(dtype=0), -2),
    (dict(rope_base=10000.0, Lmax=60000, max_seq_len=50000), -2),
    (dict(ws=FAKE, ws_bytes=64), -5),
])
def test_decode_step_rejects_invalid_arguments(lib, kw, status):
    a = dict(q_new=FAKE, k_new=FAKE, v_new=FAKE, kc=FAKE, vc=FAKE, lens=FAKE, out=FAKE, B=2, Hq=8,
             Hkv=2, Lmax=256, d=128, dtype=1, rope_base=0.0, rope_layout=0, scale=0.0,
             max_seq_len=256, splits=0, ws=FAKE, ws_bytes=1 << 24)
    a.update(kw)
    rc = lib.csattn_attn_decode_step(a["q_new"], a["k_new"], a["v_new"], a["kc"], a["vc"],
                                     a["lens"], a["out"], a["B"], a["Hq"], a["Hkv"], a["Lmax"],
                                     a["d"], a["dtype"], a["rope_base"], a["rope_layout"],
                                     a["scale"], a["max_seq_len"], a["splits"], a["ws"],
                                     a["ws_bytes"], None)
    assert rc == status, lib.csattn_last_error()
    assert b"attn_decode_step" in lib.csattn_last_error()


@pytest.mark.parametrize("kw,status", [
    (dict(lse=None), -1),
    (dict(T=0), -1),
    (dict(Hq=6, Hkv=4), -1),
    (dict(dtype=7), -1),
    (dict(d=32), -2),
    (dict(dtype=0, d=48), -2),
    (dict(dtype=0, d=256), -2),
    (dict(causal=3), -1),
    (dict(dq=FAKE + 4), -1),
    (dict(rope_base=10000.0, T=50000), -2),
    (dict(dtype=0, rope_base=10000.0, T=50000), -2),
    (dict(ws=None, ws_bytes=0), -5),
])
def test_bwd_rejects_invalid_arguments(lib, kw, status):
    a = dict(q=FAKE, k=FAKE, v=FAKE, out=FAKE, dout=FAKE, lse=FAKE, dq=FAKE, dk=FAKE, dv=FAKE,
             B=1, Hq=4, Hkv=2, T=64, d=128, dtype=1, causal=1, rope_base=0.0, rope_layout=0,
             scale=0.0, ws=FAKE, ws_bytes=1 << 24)
    a.update(kw)
    rc = lib.csattn_attn_bwd(a["q"], a["k"], a["v"], a["out"], a["dout"], a["lse"], a["dq"],
                             a["dk"], a["dv"], a["B"], a["Hq"], a["Hkv"], a["T"], a["d"],
                             a["dtype"], a["causal"], a["rope_base"], a["rope_layout"],
                             a["scale"], a["ws"], a["ws_bytes"], None)
    assert rc == status, lib.csattn_last_error()


def test_bwd_workspace_size(lib):
    rows = 4 * 32 * 4096
    al = lambda x: (x + 255) // 256 * 256  # noqa: E731
    assert lib.csattn_bwd_workspace_size(4, 32, 8, 4096, 128, 1, 0.0) == al(rows * 4)
    assert lib.csattn_bwd_workspace_size(4, 32, 8, 4096, 128, 1, 10000.0) == \
        al(rows * 4) + al(rows * 128 * 2) + al(4 * 8 * 4096 * 128 * 2)
    assert lib.csattn_bwd_workspace_size(4, 32, 8, 4096, 128, 0, 0.0) == al(rows * 4)
    assert lib.csattn_bwd_workspace_size(4, 32, 8, 4096, 128, 0, 10000.0) == \
        al(rows * 4) + al(rows * 128 * 4) + al(4 * 8 * 4096 * 128 * 4)
    assert lib.csattn_bwd_workspace_size(4, 32, 8, 4096, 128, 7, 10000.0) == 0
    assert lib.csattn_bwd_workspace_size(0, 32, 8, 4096, 128, 1, 10000.0) == 0


@pytest.mark.parametrize("kw,status", [
    (dict(dout=None), -1),
    (dict(Tq=0), -1),
    (dict(Tk=0), -1),
    (dict(q_offset=-1), -1),
    (dict(Hq=6, Hkv=4), -1),
    (dict(causal=2), -1),
    (dict(rope_layout=5), -1),
    (dict(rope_base=10000.0, rope_layout=0x100), -2),
    (dict(d_v=32), -2),
    (dict(d=256), -2),
    (dict(dtype=0, d_v=48), -2),
    (dict(q_offset=1 << 24), -2),
    (dict(rope_base=10000.0, q_offset=49100, Tq=100), -2),
    (dict(rope_base=10000.0, Tk=50000), -2),
    (dict(dk=FAKE + 8), -1),
    (dict(ws=FAKE, ws_bytes=512), -5),
])
def test_bwd_ext_rejects_invalid_arguments(lib, kw, status):
    a = dict(q=FAKE, k=FAKE, v=FAKE, out=FAKE, dout=FAKE, lse=FAKE, dq=FAKE, dk=FAKE, dv=FAKE,
             B=1, Hq=4, Hkv=2, Tq=64, Tk=192, q_offset=128, d=128, d_v=64, dtype=1, causal=1,
             rope_base=0.0, rope_layout=0, scale=0.0, ws=FAKE, ws_bytes=1 << 24)
    a.update(kw)
    rc = lib.csattn_attn_bwd_ext(a["q"], a["k"], a["v"], a["out"], a["dout"], a["lse"], a["dq"],
                                 a["dk"], a["dv"], a["B"], a["Hq"], a["Hkv"], a["Tq"], a["Tk"],
                                 a["q_offset"], a["d"], a["d_v"], a["dtype"], a["causal"],
                                 a["rope_base"], a["rope_layout"], a["scale"], a["ws"],
                                 a["ws_bytes"], None)
    assert rc == status, lib.csattn_last_error()
    assert b"attn_bwd_ext" in lib.csattn_last_error()


def test_bwd_ext_workspace_size(lib):
    al = lambda x: (x + 255) // 256 * 256  # noqa: E731
    qrows = 2 * 8 * 300
    assert lib.csattn_bwd_ext_workspace_size(2, 8, 2, 300, 1000, 64, 1, 0.0) == al(qrows * 4)
    assert lib.csattn_bwd_ext_workspace_size(2, 8, 2, 300, 1000, 64, 1, 10000.0) == \
        al(qrows * 4) + al(qrows * 64 * 2) + al(2 * 2 * 1000 * 64 * 2)
    assert lib.csattn_bwd_ext_workspace_size(2, 8, 2, 300, 1000, 32, 0, 10000.0) == \
        al(qrows * 4) + al(qrows * 32 * 4) + al(2 * 2 * 1000 * 32 * 4)
    assert lib.csattn_bwd_ext_workspace_size(2, 8, 2, 300, 0, 64, 1, 0.0) == 0
    for T in (1, 77, 4096):  # the square call's size is the ext size at Tq = Tk = T
        assert lib.csattn_bwd_workspace_size(3, 8, 2, T, 128, 1, 10000.0) == \
            lib.csattn_bwd_ext_workspace_size(3, 8, 2, T, T, 128, 1, 10000.0)


@pytest.mark.parametrize("kw,status", [
    (dict(v=None), -1),
    (dict(Hq=6, Hkv=4), -1),
    (dict(dv=32), -2),
    (dict(dv=256), -2),
    (dict(d=96), -2),
    (dict(dtype=0), -2),
    (dict(max_seq_len=0), -1),
    (dict(out=FAKE + 2), -1),
    (dict(ws=FAKE, ws_bytes=64), -5),
])
def test_decode_ext_rejects_invalid_arguments(lib, kw, status):
    a = dict(q=FAKE, k=FAKE, v=FAKE, lens=FAKE, out=FAKE, B=2, Hq=8, Hkv=2, Lmax=512, d=128,
             dv=64, dtype=1, scale=0.0, max_seq_len=512, splits=4, ws=FAKE, ws_bytes=1 << 24)
    a.update(kw)
    rc = lib.csattn_attn_decode_ext(a["q"], a["k"], a["v"], a["lens"], a["out"], a["B"], a["Hq"],
                                    a["Hkv"], a["Lmax"], a["d"], a["dv"], a["dtype"], a["scale"],
                                    a["max_seq_len"], a["splits"], a["ws"], a["ws_bytes"], None)
    assert rc == status, lib.csattn_last_error()
    assert b"attn_decode_ext" in lib.csattn_last_error()


@pytest.mark.parametrize("kw,status", [
    (dict(x=None), -1),
    (dict(T=0), -1),
    (dict(dtype=7), -1),
    (dict(d=32), -2),
    (dict(dtype=0, d=48), -2),
    (dict(dtype=0, d=256), -2),
    (dict(base=0.0), -1),
    (dict(base=float("nan")), -1),
    (dict(layout=3), -1),
    (dict(T=50000), -2),
    (dict(xr=FAKE + 8), -1),
    (dict(xr=FAKE + 64), -1),               # overlaps x
    (dict(dtype=0, d=16, xr=FAKE + 256), -1),  # fp32 rows are 4-byte elements: overlap
])
def test_rope_rotate_rejects_invalid_arguments(lib, kw, status):
    a = dict(x=FAKE, xr=FAKE + (1 << 24), B=1, H=2, T=64, d=128, dtype=1, base=10000.0,
             layout=0)
    a.update(kw)
    rc = lib.csattn_rope_rotate(a["x"], a["xr"], a["B"], a["H"], a["T"], a["d"], a["dtype"],
                                a["base"], a["layout"], None)
    assert rc == status, lib.csattn_last_error()
    assert b"rope_rotate" in lib.csattn_last_error()


def test_selftest_rejects_bad_limit(lib):
    assert lib.csattn_selftest_bounded_wait(0, None) == -1
    assert lib.csattn_selftest_bounded_wait(2000000, None) == -1


def test_product_path_does_not_import_oracle():
    pkg = os.path.join(ROOT, "transformer_causal_self_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                with open(os.path.join(dirpath, f)) as fh:
                    src = fh.read()
                assert "oracle" not in re.findall(r"^\s*(?:from|import)\s+(\w+)", src, re.M), f


def test_prefill_paged_workspace_size(lib):
    al = lambda x: (x + 255) // 256 * 256  # noqa: E731
    assert lib.csattn_prefill_paged_workspace_size(4, 8, 128, 32, 128) == 0
    assert lib.csattn_prefill_paged_workspace_size(4, 8, 64, 32, 128) == 0
    lpad = (100 * 16 + 127) // 128 * 128
    assert lib.csattn_prefill_paged_workspace_size(4, 8, 16, 100, 128) == \
        2 * al(4 * 8 * lpad * 128 * 2) + al(16)
    assert lib.csattn_prefill_paged_workspace_size(0, 8, 16, 100, 128) == 0
