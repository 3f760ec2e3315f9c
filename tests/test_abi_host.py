"""The C-ABI library on the host: it loads, exports every symbol the header
declares, and rejects bad arguments synchronously without touching a GPU."""
import ctypes
import os
import re
import subprocess

import pytest

import sequence_depth_attention_gb300 as moda
from sequence_depth_attention_gb300 import binding
from sequence_depth_attention_gb300 import build as mbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moda.h")

OK, INVALID, UNSUPPORTED, MISALIGNED, CUDA, TIMEOUT, NO_DEVICE = range(7)


@pytest.fixture(scope="module")
def lib():
    mbuild.build()
    return binding.load()


def header_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"MODA_API\s+[\w\s\*]+?\b(moda_\w+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert header_functions() == sorted(binding.EXPORTS)


def test_library_exports_every_header_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", binding.library_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT\s+(moda_\w+)", out))
    missing = set(header_functions()) - exported
    assert not missing, f"not exported: {missing}"
    # nothing but the ABI leaks out of the library
    assert exported == set(header_functions())


def test_status_strings(lib):
    names = ["MODA_OK", "MODA_ERR_INVALID_ARG", "MODA_ERR_UNSUPPORTED", "MODA_ERR_MISALIGNED",
             "MODA_ERR_CUDA", "MODA_ERR_TIMEOUT", "MODA_ERR_NO_DEVICE"]
    for code, name in enumerate(names):
        assert moda.moda_status_string(code) == name
    assert moda.moda_status_string(99) == "MODA_ERR_UNKNOWN"


# Fake device addresses: validation must reject before dereferencing anything.
A = 0x10000000
B = 0x20000000
C = 0x30000000
D = 0x40000000
E = 0x50000000
O = 0x60000000
LSE = 0x70000000


def fwd(lib, q=A, k=B, v=C, kd=D, vd=E, T=128, Hq=4, Hk=2, d=64, L=4, scale=0.125, o=O, lse=LSE):
    return lib.moda_fwd(q, k, v, kd, vd, T, Hq, Hk, d, L, scale, o, lse, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), INVALID), (dict(k=None), INVALID), (dict(v=None), INVALID),
    (dict(o=None), INVALID), (dict(kd=None), INVALID), (dict(vd=None), INVALID),
    (dict(T=0), INVALID), (dict(T=-5), INVALID), (dict(L=-1), INVALID),
    (dict(Hq=5, Hk=2), INVALID), (dict(Hk=0), INVALID),
    (dict(scale=float("nan")), INVALID), (dict(scale=float("inf")), INVALID),
    (dict(scale=0.0), INVALID), (dict(scale=-0.125), INVALID),
    (dict(d=96), UNSUPPORTED), (dict(d=256), UNSUPPORTED),
    (dict(Hq=6, Hk=2), UNSUPPORTED), (dict(Hq=64, Hk=2), UNSUPPORTED),
    (dict(T=(1 << 24) + 1), UNSUPPORTED), (dict(L=1025), UNSUPPORTED),
    (dict(q=A + 8), MISALIGNED), (dict(kd=D + 2), MISALIGNED), (dict(o=O + 4), MISALIGNED),
    (dict(lse=LSE + 4), MISALIGNED),
    (dict(o=A), INVALID),                       # o aliases q
    (dict(lse=B + 64), INVALID),                # lse inside k
    (dict(lse=O + 1024), INVALID),              # lse inside o
])
def test_fwd_rejects(lib, kw, code):
    assert fwd(lib, **kw) == code
    assert lib.moda_last_error_detail().decode() != ""


def fwd_lm(lib, q=A, k=B, v=C, kd=D, vd=E, T=128, Hq=4, Hk=2, d=64, L=4, scale=0.125, o=O, lse=LSE):
    return lib.moda_fwd_layer_major(q, k, v, kd, vd, T, Hq, Hk, d, L, scale, o, lse, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), INVALID), (dict(kd=None), INVALID), (dict(T=0), INVALID),
    (dict(d=96), UNSUPPORTED), (dict(Hq=6, Hk=2), UNSUPPORTED), (dict(L=1025), UNSUPPORTED),
    (dict(vd=E + 2), MISALIGNED), (dict(o=A), INVALID), (dict(lse=D + 64), INVALID),
])
def test_fwd_layer_major_rejects(lib, kw, code):
    # the layer-major forward validates exactly like moda_fwd
    assert fwd_lm(lib, **kw) == code
    assert lib.moda_last_error_detail().decode() != ""


WS = 0x80000000  # fake device workspace, 256-byte aligned


def fwd_host(lib, q=A, k=B, v=C, kd=D, vd=E, T=128, Hq=4, Hk=2, d=64, L=4, scale=0.125, o=O,
             lse=LSE, ws=WS, nbytes=None):
    if nbytes is None:
        nbytes = lib.moda_fwd_host_workspace_bytes(T, Hq, Hk, d, L)
    return lib.moda_fwd_layer_major_host(q, k, v, kd, vd, T, Hq, Hk, d, L, scale, o, lse, ws,
                                         nbytes, None)


def test_fwd_host_workspace_bytes(lib):
    # q 64 KB, k and v 32 KB, kd and vd 128 KB, o 64 KB, lse 2 KB, each region
    # on a 256-byte boundary
    assert lib.moda_fwd_host_workspace_bytes(128, 4, 2, 64, 4) == 460800
    # 384-byte q, k, v and o each take two 256-byte units, kd and vd none
    assert lib.moda_fwd_host_workspace_bytes(3, 1, 1, 64, 0) == 512 * 4 + 256
    for bad in ((0, 4, 2, 64, 4), (128, 0, 2, 64, 4), (128, 4, 2, 64, -1)):
        assert lib.moda_fwd_host_workspace_bytes(*bad) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(ws=None), INVALID), (dict(ws=WS + 16), MISALIGNED), (dict(nbytes=460799), INVALID),
    (dict(q=None), INVALID), (dict(o=None), INVALID), (dict(kd=None), INVALID),
    (dict(T=0), INVALID), (dict(scale=float("nan")), INVALID), (dict(d=96), UNSUPPORTED),
    (dict(Hq=6, Hk=2), UNSUPPORTED), (dict(L=1025), UNSUPPORTED),
    (dict(lse=O + 1024), INVALID),             # lse inside o
    (dict(o=WS + 4096), INVALID),              # a host buffer inside the workspace
])
def test_fwd_layer_major_host_rejects(lib, kw, code):
    assert fwd_host(lib, **kw) == code
    assert lib.moda_last_error_detail().decode() != ""


def test_fwd_layer_major_host_without_gpu_reports_no_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert fwd_host(lib) == NO_DEVICE
    assert fwd_host(lib, kd=None, vd=None, L=0, lse=None) == NO_DEVICE


def fwd_cc(lib, q=A, k=B, v=C, kd=D, vd=E, T=128, Hq=4, Hk=2, d=64, L=4, scale=0.125, o=O, lse=LSE):
    return lib.moda_fwd_depth_cc(q, k, v, kd, vd, T, Hq, Hk, d, L, scale, o, lse, None)


@pytest.mark.parametrize("kw,code", [
    (dict(lse=None), INVALID), (dict(q=None), INVALID), (dict(d=96), UNSUPPORTED),
    (dict(Hq=6, Hk=2), UNSUPPORTED), (dict(kd=D + 2), MISALIGNED), (dict(o=A), INVALID),
])
def test_fwd_depth_cc_rejects(lib, kw, code):
    # the CUDA-core depth variant validates exactly like moda_fwd, and needs lse
    assert fwd_cc(lib, **kw) == code


def test_fwd_l0_accepts_null_depth(lib):
    # L = 0 with NULL kd/vd passes validation; without a GPU it stops at the
    # device check, with one it would run (covered by the GPU tests).
    rc = fwd(lib, kd=None, vd=None, L=0)
    assert rc in (OK, NO_DEVICE)


def test_fwd_without_gpu_reports_no_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert fwd(lib) == NO_DEVICE


@pytest.mark.parametrize("args,code", [
    ((A, B, -1, 8, 2, 64), INVALID), ((A, B, 2, 0, 2, 64), INVALID),
    ((A, B, 2, 8, 0, 64), INVALID), ((A, B, 2, 8, 2, 80), UNSUPPORTED),
    ((None, B, 2, 8, 2, 64), INVALID), ((A, None, 2, 8, 2, 64), INVALID),
    ((A + 4, B, 2, 8, 2, 64), MISALIGNED), ((A, A + 512, 2, 8, 2, 64), INVALID),
])
def test_pack_rejects(lib, args, code):
    assert lib.moda_pack_depth(*args, None) == code


def test_pack_l0_is_noop(lib):
    assert lib.moda_pack_depth(None, None, 0, 8, 2, 64, None) == OK


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(binding, "_LIB", str(tmp_path / "missing.so"))
    monkeypatch.setattr(binding, "_lib", None)
    with pytest.raises(binding.ModaError):
        binding.load()


def test_product_package_does_not_import_oracle():
    pkg = os.path.join(ROOT, "sequence_depth_attention_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".h", ".cc", ".c")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(from|import)\s+oracle\b", text, re.M), f
                assert "moda_oracle" not in text, f


@pytest.mark.parametrize("ms", [0, -1, 5001])
def test_selftest_rejects_timeout(lib, ms):
    assert lib.moda_selftest_wait_timeout(ms, None) == INVALID


@pytest.mark.parametrize("args,code", [
    ((A, B, 0, 2, 64, 4, 0), INVALID), ((A, B, 8, 2, 64, 0, 0), INVALID),
    ((A, B, 8, 2, 64, 4, 4), INVALID), ((A, B, 8, 2, 64, 4, -1), INVALID),
    ((A, B, 8, 2, 96, 4, 0), UNSUPPORTED), ((A, B, 8, 2, 64, 2000, 0), UNSUPPORTED),
    ((None, B, 8, 2, 64, 4, 0), INVALID), ((A + 8, B, 8, 2, 64, 4, 0), MISALIGNED),
    ((A, A + 256, 8, 2, 64, 4, 0), INVALID),
])
def test_depth_write_rejects(lib, args, code):
    assert lib.moda_depth_write(*args, None) == code


def _proj(lib, x=A, wk=B, wv=C, T=8, Dm=128, Hk=2, d=64, L=4, slot=1, kd=D, vd=E):
    lib.moda_kv_proj_write.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 6 + [ctypes.c_void_p] * 3
    return lib.moda_kv_proj_write(x, wk, wv, T, Dm, Hk, d, L, slot, kd, vd, None)


@pytest.mark.parametrize("kw,code", [
    (dict(x=None), INVALID), (dict(vd=None), INVALID), (dict(T=0), INVALID), (dict(L=0), INVALID),
    (dict(slot=4), INVALID), (dict(slot=-1), INVALID), (dict(Dm=96), UNSUPPORTED),
    (dict(d=96), UNSUPPORTED), (dict(L=1025, slot=0), UNSUPPORTED), (dict(wk=B + 8), MISALIGNED),
    (dict(kd=A), INVALID), (dict(vd=D + 64), INVALID),
])
def test_kv_proj_rejects(lib, kw, code):
    assert _proj(lib, **kw) == code


def test_decode_workspace_formula(lib):
    lib.moda_decode_workspace_bytes.restype = ctypes.c_size_t
    # (splits + 1) partials of (d + 2) floats per head; splits <= ceil(T/64), capped at 128
    assert lib.moda_decode_workspace_bytes(1, 16, 128) == 2 * 16 * 130 * 4
    assert lib.moda_decode_workspace_bytes(640, 16, 128) == 11 * 16 * 130 * 4
    assert lib.moda_decode_workspace_bytes(65536, 16, 128) == 129 * 16 * 130 * 4
    assert lib.moda_decode_workspace_bytes(0, 16, 128) == 0


def _dec(lib, q=A, kc=B, vc=C, kt=D, vt=E, stride=4 * 64, T=100, Hq=4, Hk=2, d=64, L=4,
         scale=0.125, o=O, lse=LSE, ws=0x78000000, wsb=1 << 20):
    lib.moda_decode.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_longlong] + [ctypes.c_int] * 5 + [
        ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
        ctypes.c_void_p]
    return lib.moda_decode(q, kc, vc, kt, vt, stride, T, Hq, Hk, d, L, scale, o, lse, ws, wsb, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), INVALID), (dict(ws=None), INVALID), (dict(T=0), INVALID),
    (dict(kt=None), INVALID), (dict(stride=4 * 64 - 8), INVALID), (dict(stride=4 * 64 + 3), INVALID),
    (dict(wsb=16), INVALID), (dict(d=96), UNSUPPORTED), (dict(Hq=6, Hk=2), UNSUPPORTED),
    (dict(q=A + 2), MISALIGNED), (dict(o=B), INVALID), (dict(scale=-1.0), INVALID),
])
def test_decode_rejects(lib, kw, code):
    assert _dec(lib, **kw) == code


# ---- bounded depth cache entry points
def test_depth_mass_workspace_formula(lib):
    # one [L] partial per CTA: per KV head, ceil(T / 4) CTAs (four positions,
    # one per warp, at least) up to 2048 CTAs over all heads
    assert lib.moda_depth_mass_workspace_bytes(64, 4, 48) == 16 * 4 * 48 * 4
    assert lib.moda_depth_mass_workspace_bytes(65536, 4, 48) == 512 * 4 * 48 * 4
    assert lib.moda_depth_mass_workspace_bytes(65, 2, 3) == 17 * 2 * 3 * 4
    assert lib.moda_depth_mass_workspace_bytes(65536, 4096, 1) == 1 * 4096 * 1 * 4
    assert lib.moda_depth_mass_workspace_bytes(0, 4, 48) == 0


def _mass(lib, q=A, kd=B, lse=C, T=100, Hq=4, Hk=2, d=64, L=4, scale=0.125, mass=D, ws=E,
          wsb=1 << 20):
    return lib.moda_depth_mass(q, kd, lse, T, Hq, Hk, d, L, scale, mass, ws, wsb, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), INVALID), (dict(ws=None), INVALID), (dict(T=0), INVALID), (dict(L=0), INVALID),
    (dict(Hq=5, Hk=2), INVALID), (dict(scale=0.0), INVALID), (dict(wsb=16), INVALID),
    (dict(d=96), UNSUPPORTED), (dict(Hq=6, Hk=2), UNSUPPORTED), (dict(L=1025), UNSUPPORTED),
    (dict(lse=C + 4), MISALIGNED), (dict(mass=A), INVALID), (dict(ws=C), INVALID),
])
def test_depth_mass_rejects(lib, kw, code):
    assert _mass(lib, **kw) == code


def _admit(lib, ages=A, mass=B, Hk=2, S=4, recent=1, new_age=5, slot=C):
    return lib.moda_depth_cache_admit(ages, mass, Hk, S, recent, new_age, slot, None)


@pytest.mark.parametrize("kw,code", [
    (dict(ages=None), INVALID), (dict(slot=None), INVALID), (dict(S=0), INVALID),
    (dict(Hk=0), INVALID), (dict(recent=-1), INVALID), (dict(new_age=-1), INVALID),
    (dict(S=1025), UNSUPPORTED), (dict(slot=C + 2), MISALIGNED), (dict(slot=A + 4), INVALID),
])
def test_cache_admit_rejects(lib, kw, code):
    assert _admit(lib, **kw) == code


@pytest.mark.parametrize("args,code", [
    ((A, B, 0, 2, 64, 4, C), INVALID), ((A, B, 8, 2, 64, 0, C), INVALID),
    ((A, B, 8, 2, 64, 4, None), INVALID), ((A, B, 8, 2, 96, 4, C), UNSUPPORTED),
    ((A, B, 8, 2, 64, 2000, C), UNSUPPORTED), ((A + 8, B, 8, 2, 64, 4, C), MISALIGNED),
    ((A, B, 8, 2, 64, 4, C + 1), MISALIGNED), ((A, A + 256, 8, 2, 64, 4, C), INVALID),
])
def test_depth_write_at_rejects(lib, args, code):
    assert lib.moda_depth_write_at(*args, None) == code


def _dec_strided(lib, q=A, kc=B, vc=C, kt=D, vt=E, slot=100 * 2 * 64, hks=64, T=100, Hq=4, Hk=2,
                 d=64, L=4, scale=0.125, o=O, lse=LSE, ws=0x78000000, wsb=1 << 20):
    lib.moda_decode_strided.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_longlong] * 2 + [
        ctypes.c_int] * 5 + [ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                             ctypes.c_size_t, ctypes.c_void_p]
    return lib.moda_decode_strided(q, kc, vc, kt, vt, slot, hks, T, Hq, Hk, d, L, scale, o, lse, ws,
                                   wsb, None)


@pytest.mark.parametrize("kw,code", [
    (dict(slot=0), INVALID), (dict(slot=32), INVALID), (dict(slot=68), INVALID),
    (dict(hks=32), INVALID), (dict(hks=66), INVALID), (dict(q=None), INVALID),
    (dict(d=96), UNSUPPORTED), (dict(L=1025), UNSUPPORTED), (dict(kt=D + 2), MISALIGNED),
    (dict(o=D + 12800 * 2), INVALID),   # o inside the strided depth slots
])
def test_decode_strided_rejects(lib, kw, code):
    # the strided decode validates its strides and otherwise as moda_decode
    assert _dec_strided(lib, **kw) == code
    assert lib.moda_last_error_detail().decode() != ""
