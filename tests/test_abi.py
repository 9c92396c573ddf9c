"""The C-ABI library loads, exports every entry point its header declares, and
rejects bad arguments on the host before touching CUDA (CPU only: every call
here fails validation, so nothing is enqueued)."""
import ctypes
import os
import re

import pytest

import dit_modulate_absmax_gb300 as pkg
from dit_modulate_absmax_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, NULL, ALIGN, SHAPE, UNSUP = 0, 1, 2, 3, 4


@pytest.fixture(scope="module")
def L():
    B.build()
    return pkg.lib()


def _declared():
    text = open(os.path.join(ROOT, "include", "h3fp4.h")).read()
    return sorted(set(re.findall(r"H3FP4_API\s+[\w\s\*]*?\b(h3fp4_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ("h3fp4_modulate_absmax", "h3fp4_modulate_pack", "h3fp4_swiglu_pack", "h3fp4_gemm"):
        assert n in names
    assert set(names) <= set(pkg._SIGNATURES)


def test_library_exports_every_declared_symbol(L):
    for name in _declared():
        assert hasattr(L, name), name
    out = os.popen(f"nm -D --defined-only {pkg.LIB_PATH}").read()
    exported = set(re.findall(r"\bT (h3fp4_\w+)", out))
    assert set(_declared()) <= exported


def test_header_is_plain_c_and_the_library_links_from_c(L, tmp_path):
    """A C11 program (gcc, -Wall -Werror -pedantic) includes the header, links
    libh3fp4.so directly and calls entry points that need no GPU."""
    exe = tmp_path / "abi_c_check"
    src = os.path.join(ROOT, "tests", "helpers", "abi_c_check.c")
    libdir = os.path.dirname(pkg.LIB_PATH)
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
           src, "-o", str(exe), f"-L{libdir}", "-l:libh3fp4.so", f"-Wl,-rpath,{libdir}"]
    import subprocess
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr


def test_status_strings_and_build_info(L):
    assert pkg.lib().h3fp4_status_string(0) == b"ok"
    assert pkg.lib().h3fp4_status_string(3) == b"invalid shape"
    assert pkg.lib().h3fp4_status_string(99) == b"unknown status"
    info = pkg.h3fp4_build_info()
    assert "sm_103a" in info and "nvcc" in info


F = 0x10000        # a fake, 16-byte aligned "device" address (never dereferenced)


def _offs(*v):
    return (ctypes.c_int32 * len(v))(*v)


def test_modulate_absmax_validation(L):
    f = L.h3fp4_modulate_absmax
    good = dict(x=F, ldx=256, m=10, d=256, sh=F, sc=F, ldm=256, off=_offs(0, 10), n=1, ts=F, scr=F)

    def call(**kw):
        a = {**good, **kw}
        return f(a["x"], a["ldx"], a["m"], a["d"], a["sh"], a["sc"], a["ldm"], a["off"], a["n"], a["ts"], a["scr"], None)

    assert call(x=None) == NULL
    assert call(x=None, m=0, off=_offs(0, 0)) != NULL      # nothing is read from x when m == 0
    assert call(ts=None) == NULL
    assert call(scr=None) == NULL
    assert call(off=None) == NULL
    assert call(d=100) == SHAPE            # not a multiple of 256
    assert call(m=-1) == SHAPE
    assert call(ldx=128) == SHAPE          # ldx < d
    assert call(x=F + 8) == ALIGN
    assert call(ldx=260) == ALIGN
    assert call(off=_offs(0, 9), n=1) == SHAPE          # last offset != m
    assert call(off=_offs(1, 10), n=1) == SHAPE         # first offset != 0
    assert call(off=_offs(0, 6, 4, 10), n=3) == SHAPE   # not monotone
    assert call(n=0) == SHAPE
    assert call(n=17) == SHAPE


def test_modulate_pack_validation(L):
    f = L.h3fp4_modulate_pack
    off = _offs(0, 10)
    assert f(F, 256, 10, 8, 256, F, F, 256, off, 1, F, F, F, None) == SHAPE        # m_pad < m
    assert f(F, 256, 10, 24, 256, F, F, 256, off, 1, F, F, F, None) == SHAPE       # m_pad not a multiple of 16
    assert f(F, 256, 10, 16, 256, F, F, 256, off, 1, None, F, F, None) == NULL
    assert f(F, 256, 10, 16, 256, F, F, 256, off, 1, F, None, F, None) == NULL
    assert f(F, 256, 10, 16, 256, F, F, 256, off, 1, F, F, F + 4, None) == ALIGN


def test_swiglu_pack_validation(L):
    f = L.h3fp4_swiglu_pack
    assert f(None, 256, F, 256, 10, 16, 256, F, F, F, F, None, None) == NULL
    assert f(F, 256, F, 256, 10, 16, 300, F, F, F, F, None, None) == SHAPE
    assert f(F, 256, F, 256, 10, 16, 256, F, F, F, F, F + 2, None) == ALIGN
    assert f(F, 256, F, 256, 10, 4, 256, F, F, F, F, None, None) == SHAPE
    assert f(F, 256, F, 256, 10, 20, 256, F, F, F, F, None, None) == SHAPE      # m_pad not a multiple of 16


def test_swiglu_pack_noalloc_validation(L):
    f = L.h3fp4_swiglu_pack_noalloc
    assert f(None, 256, F, 256, 10, 16, 256, F, F, F, None) == NULL
    assert f(F, 256, F, 256, 10, 16, 300, F, F, F, None) == SHAPE               # f not a multiple of 256
    assert f(F, 256, F, 256, 10, 4, 256, F, F, F, None) == SHAPE                # m_pad < m
    assert f(F, 256, F, 256, 10, 20, 256, F, F, F, None) == SHAPE               # m_pad not a multiple of 16
    big = pkg.NOALLOC_MAX_ELEMENTS // 256 + 1
    assert f(F, 256, F, 256, big, -(-big // 16) * 16, 256, F, F, F, None) == SHAPE   # beyond the static scratch


def test_modulate_produce_validation(L):
    f = L.h3fp4_modulate_produce
    offs = (ctypes.c_int32 * 2)(0, 10)
    assert f(None, 256, 10, 16, 256, F, F, 256, offs, 1, F, F, F, F, None) == NULL
    assert f(F, 256, 10, 16, 256, F, F, 256, offs, 1, None, F, F, F, None) == NULL     # tensor scale
    assert f(F, 256, 10, 16, 300, F, F, 256, offs, 1, F, F, F, F, None) == SHAPE
    assert f(F, 256, 10, 4, 256, F, F, 256, offs, 1, F, F, F, F, None) == SHAPE       # m_pad < m
    assert f(F, 256, 10, 40, 256, F, F, 256, offs, 1, F, F, F, F, None) == SHAPE      # m_pad not a multiple of 16
    assert f(F, 256, 10, 16, 256, F, F, 256, (ctypes.c_int32 * 2)(0, 9), 1, F, F, F, F, None) == SHAPE


def test_quantize_pack_validation(L):
    f = L.h3fp4_quantize_pack
    assert f(None, 256, 10, 16, 256, F, F, F, F, None) == NULL
    assert f(F, 256, 10, 16, 300, F, F, F, F, None) == SHAPE       # d not a multiple of 256
    assert f(F, 200, 10, 16, 256, F, F, F, F, None) == SHAPE       # ldx < d
    assert f(F + 2, 256, 10, 16, 256, F, F, F, F, None) == ALIGN
    assert f(F, 256, 10, 4, 256, F, F, F, F, None) == SHAPE         # m_pad < m
    assert f(F, 256, 10, 17, 256, F, F, F, F, None) == SHAPE        # m_pad not a multiple of 16


def test_gemm_validation(L):
    f = L.h3fp4_gemm

    def call(m=300, m_pad=320, n=384, k=256, ldc=384, c=F, cfg=None):
        return f(F, F, F, F, F, F, c, ldc, m, m_pad, n, k, cfg, None)

    assert call(c=None) == NULL
    assert call(k=128) == SHAPE
    assert call(n=100) == SHAPE
    assert call(m=400) == SHAPE            # m > m_pad
    assert call(m_pad=310) == SHAPE        # m_pad not a multiple of 16
    assert call(ldc=200) == SHAPE
    assert call(ldc=388) == ALIGN
    assert call(c=F + 2) == ALIGN
    bad = pkg.GemmConfig(-1, 0, 0, 0)
    assert call(cfg=ctypes.byref(bad)) == UNSUP
    bad = pkg.GemmConfig(0, 3, 0, 0)
    assert call(cfg=ctypes.byref(bad)) == UNSUP
    for kernel in (2, 3, 5):               # kernels are 0 (default), 1 and 4
        bad = pkg.GemmConfig(0, 0, kernel, 0)
        assert call(cfg=ctypes.byref(bad)) == UNSUP


def test_gemm_gated_residual_validation(L):
    f = L.h3fp4_gemm_gated_residual
    offs = (ctypes.c_int32 * 3)(0, 200, 300)

    def call(gate=F, ld_gate=384, residual=F + 4096 * 1024, ldr=384, out=F, ldo=384, nseg=2, off=offs, cfg=None):
        return f(F, F, F, F, F, F, gate, ld_gate, off, nseg, residual, ldr, out, ldo, 300, 320, 384, 256, cfg, None)

    assert call(gate=None) == NULL
    assert call(residual=None) == NULL
    assert call(ld_gate=256) == SHAPE
    assert call(ldr=256) == SHAPE
    assert call(gate=F + 2) == ALIGN
    assert call(ldr=388) == ALIGN
    assert call(off=(ctypes.c_int32 * 3)(0, 250, 200)) == SHAPE          # offsets must not decrease
    assert call(residual=F + 64) == UNSUP                                 # partial overlap with the output
    assert call(cfg=ctypes.byref(pkg.GemmConfig(0, 0, 3, 0))) == UNSUP     # no such kernel


def test_failure_detection_entry_points_validation(L):
    f = L.h3fp4_diag_producer_barrier_timeout
    assert f(None, 256, 10, 16, 256, F, F, F, F, 1000, None) == NULL
    assert f(F, 256, 10, 16, 256, F, F, F, F, 0, None) == SHAPE              # limit must be >= 1 us
    assert f(F, 256, 10, 16, 256, F, F, F, F, 2000001, None) == SHAPE        # and <= 2 s
    assert f(F, 256, 10, 20, 256, F, F, F, F, 1000, None) == SHAPE           # m_pad not a multiple of 16
    g = L.h3fp4_diag_gemm_wait_timeout
    assert g(F, F, F, F, F, F, None, 384, 300, 320, 384, 256, 1000, None) == NULL
    assert g(F, F, F, F, F, F, F, 384, 300, 320, 384, 128, 1000, None) == SHAPE     # k not a multiple of 256
    assert g(F, F, F, F, F, F, F, 384, 300, 320, 384, 256, 0, None) == SHAPE


def test_swizzle_and_device_error_validation(L):
    assert L.h3fp4_swizzle_scales(None, 10, 16, 16, F, None) == NULL
    assert L.h3fp4_swizzle_scales(F, 10, 6, 16, F, None) == SHAPE
    assert L.h3fp4_swizzle_scales(F, 10, 16, 8, F, None) == SHAPE
    assert L.h3fp4_swizzle_scales(F, 10, 16, 16, F + 1, None) == ALIGN
    assert L.h3fp4_device_error(None) == NULL


def test_python_binding_raises_on_error(L):
    with pytest.raises(pkg.H3FP4Error) as e:
        pkg.h3fp4_gemm(F, F, F, F, F, F, None, 384, 300, 320, 384, 256)
    assert e.value.status == NULL
