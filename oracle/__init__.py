"""Plain CPU oracle for the modulation-fused NVFP4 producer and block-scaled GEMM.

TEST INFRASTRUCTURE ONLY.  The test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only callers.  Nothing here is shared
with the CUDA path (``dit_modulate_absmax_gb300``), and the CUDA path never
imports this package.

What each function computes, and the passage it follows:

* :func:`modulate` -- AdaLN modulation ``(x * (scale + 1)) + shift`` with a BF16
  rounding after every operation and per-segment shift/scale rows
  ("NVFP4 Modulation Producer Fusion", Exactness Contract).
* :func:`absmax`, :func:`tensor_scale` -- one exact global BF16 absolute maximum
  and one FP32 tensor scale ``RN_f32(amax / 2688)``
  ("NVFP4 Streaming Design", Numerical Constraint, items 1-2).
* :func:`pack` -- one E4M3 block scale per 16 values and E2M1 codes quantised
  with both scales, zero padding rows ("NVFP4 Streaming Design", Numerical
  Constraint, items 3-4; "FC2 NVFP4 Library Scheduling", Exact Operation, the
  37,810 -> 37,824 padding).
* :func:`silu_table`, :func:`swiglu` -- BF16 SwiGLU ``RN_bf16(silu(g) * u)`` with
  the correctly rounded BF16 silu ("FC2 NVFP4 Library Scheduling", Exact
  Operation / Current Baseline).
* :func:`gemm_reference` -- FP64 sum of dequantised products
  ``sum_k a_k b_k`` with ``a_k = e2m1 * e4m3 * ts_a`` (and ``b_k`` alike) plus
  ``sum_k |a_k b_k|`` for the tolerance ("NVFP4 Streaming Design", Available
  Foundation and P0; "FC2 NVFP4 Library Scheduling", Exact Operation).

Bit-level work runs in ``h3fp4_oracle.c`` (plain loops, IEEE double, one generic
rounding routine); sums of products use numpy FP64 matmul as a library step.

Parity pins: every function above is pinned by ``tests/test_oracle_pins.py``
against brute force, closed forms, a library routine (torch CPU BF16 ops,
torch float8_e4m3fn casts) or hand-derived golden values in ``tests/golden``.
NaN/Inf inputs (adversarial cases the pages list without expected bytes)
follow the formulas in IEEE arithmetic with two stated conventions -- a NaN
quotient encodes as the E4M3 NaN code 0x7F, and a zero or NaN scale product
gives zeros with y's signs -- pinned by hand-derived bytes.
"""
from __future__ import annotations

import ctypes
import functools
import os
import struct
import subprocess
from decimal import Decimal, localcontext
from fractions import Fraction

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "h3fp4_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")

# Scale-factor tiles of the GEMM's scale layout cover 128 rows.
SF_ROW_TILE = 128


def build(force: bool = False) -> str:
    """Compile the C oracle (gcc, no fast-math, no FMA contraction), with
    OpenMP over rows where the compiler supports it (serial otherwise)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]
        try:
            subprocess.check_call(base + ["-fopenmp", "-o", tmp, _SRC, "-lm"], stderr=subprocess.DEVNULL)
        except subprocess.CalledProcessError:
            subprocess.check_call(base + ["-Wno-unknown-pragmas", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_P = ctypes.c_void_p
_I64 = ctypes.c_int64


@functools.lru_cache(maxsize=None)
def lib() -> ctypes.CDLL:
    L = ctypes.CDLL(build())
    L.orc_round.restype = ctypes.c_double
    L.orc_round.argtypes = [ctypes.c_double, ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int]
    for name in ("orc_rn_bf16", "orc_rn_f32"):
        getattr(L, name).restype = ctypes.c_double
        getattr(L, name).argtypes = [ctypes.c_double]
    L.orc_bf16_value.restype = ctypes.c_double
    L.orc_bf16_value.argtypes = [ctypes.c_uint16]
    L.orc_bf16_bits.restype = ctypes.c_uint16
    L.orc_bf16_bits.argtypes = [ctypes.c_double]
    L.orc_e4m3_decode.restype = ctypes.c_double
    L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
    L.orc_e4m3_encode.restype = ctypes.c_uint8
    L.orc_e4m3_encode.argtypes = [ctypes.c_double]
    L.orc_e2m1_decode.restype = ctypes.c_double
    L.orc_e2m1_decode.argtypes = [ctypes.c_uint8]
    L.orc_e2m1_encode.restype = ctypes.c_uint8
    L.orc_e2m1_encode.argtypes = [ctypes.c_double]
    L.orc_modulate.restype = None
    L.orc_modulate.argtypes = [_P, _I64, _I64, _I64, _P, _P, _I64, _P, ctypes.c_int32, _P, _I64]
    L.orc_gated_residual.restype = None
    L.orc_gated_residual.argtypes = [_P, _I64, _P, _I64, _P, ctypes.c_int32, _P, _I64, _I64, _I64, _P, _I64]
    L.orc_swiglu.restype = None
    L.orc_swiglu.argtypes = [_P, _I64, _P, _I64, _I64, _I64, _P, _P, _I64]
    L.orc_absmax.restype = ctypes.c_uint16
    L.orc_absmax.argtypes = [_P, _I64, _I64, _I64]
    L.orc_tensor_scale.restype = ctypes.c_float
    L.orc_tensor_scale.argtypes = [ctypes.c_uint16]
    L.orc_pack.restype = None
    L.orc_pack.argtypes = [_P, _I64, _I64, _I64, _I64, ctypes.c_float, _P, _P, _I64]
    L.orc_sf_offset.restype = _I64
    L.orc_sf_offset.argtypes = [_I64, _I64, _I64]
    L.orc_swizzle_sf.restype = None
    L.orc_swizzle_sf.argtypes = [_P, _I64, _I64, _P]
    L.orc_unswizzle_sf.restype = None
    L.orc_unswizzle_sf.argtypes = [_P, _I64, _I64, _P]
    L.orc_dequant.restype = None
    L.orc_dequant.argtypes = [_P, _P, _I64, ctypes.c_float, _I64, _I64, _P]
    L.orc_set_threads.restype = None
    L.orc_set_threads.argtypes = [ctypes.c_int]
    L.orc_threads.restype = ctypes.c_int
    L.orc_threads.argtypes = []
    return L


def set_threads(n: int) -> None:
    """Threads for the C row loops (1 = the plain serial oracle)."""
    lib().orc_set_threads(int(n))


def threads() -> int:
    return int(lib().orc_threads())


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _u16(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a).view(np.uint16) if np.asarray(a).dtype != np.uint16 else a)


# ----------------------------------------------------------------------------
# Scalars and codecs
# ----------------------------------------------------------------------------
def rn_bf16(v: float) -> float:
    return lib().orc_rn_bf16(float(v))


def rn_f32(v: float) -> float:
    return lib().orc_rn_f32(float(v))


def bf16_value(bits: int) -> float:
    return lib().orc_bf16_value(int(bits) & 0xFFFF)


def bf16_bits(v: float) -> int:
    """bf16 pattern of the correctly rounded value of v (a Python float)."""
    return lib().orc_bf16_bits(rn_bf16(v))


def e4m3_encode(v: float) -> int:
    return lib().orc_e4m3_encode(float(v))


def e4m3_decode(c: int) -> float:
    return lib().orc_e4m3_decode(int(c) & 0xFF)


def e2m1_encode(v: float) -> int:
    return lib().orc_e2m1_encode(float(v))


def e2m1_decode(c: int) -> float:
    return lib().orc_e2m1_decode(int(c) & 0xF)


@functools.lru_cache(maxsize=None)
def e4m3_table() -> np.ndarray:
    return np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)


@functools.lru_cache(maxsize=None)
def e2m1_table() -> np.ndarray:
    return np.array([e2m1_decode(c) for c in range(16)], dtype=np.float64)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact values of bf16 patterns (a bf16 is the top half of an fp32)."""
    b = np.asarray(bits).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------
# Producer steps
# ----------------------------------------------------------------------------
def modulate(x, shift, scale, seg_off) -> np.ndarray:
    """y = RN_bf16(RN_bf16(x * RN_bf16(scale_s + 1)) + shift_s), row r in segment s.

    x: uint16 [m, d] bf16 patterns; shift/scale: uint16 [nseg, d];
    seg_off: int32 [nseg + 1] row offsets (0 ... m).
    """
    x = _u16(x)
    shift = _u16(shift)
    scale = _u16(scale)
    m, d = x.shape
    off = np.ascontiguousarray(np.asarray(seg_off, dtype=np.int32))
    nseg = len(off) - 1
    assert shift.shape == (nseg, d) and scale.shape == (nseg, d)
    assert off[0] == 0 and off[-1] == m and np.all(np.diff(off) >= 0)
    y = np.empty((m, d), dtype=np.uint16)
    lib().orc_modulate(_ptr(x), d, m, d, _ptr(shift), _ptr(scale), d, _ptr(off), nseg, _ptr(y), d)
    return y


def absmax(y) -> int:
    """bf16 pattern of max |y| over all (logical) rows; NaN if any NaN."""
    y = _u16(y)
    m, d = y.shape
    return int(lib().orc_absmax(_ptr(y), d, m, d))


def tensor_scale(amax_bits: int) -> float:
    """FP32 tensor scale RN_f32(amax / (6 * 448))."""
    return float(lib().orc_tensor_scale(int(amax_bits)))


def sf_rows_for(m_pad: int) -> int:
    return -(-m_pad // SF_ROW_TILE) * SF_ROW_TILE


def pack(y, m_pad: int, ts: float):
    """E2M1 QDATA [m_pad, d/2] and LOGICAL E4M3 scales [ceil128(m_pad), d/16]."""
    y = _u16(y)
    m, d = y.shape
    assert d % 16 == 0 and m_pad >= m
    rows = sf_rows_for(m_pad)
    q = np.empty((m_pad, d // 2), dtype=np.uint8)
    sf = np.empty((rows, d // 16), dtype=np.uint8)
    lib().orc_pack(_ptr(y), d, m, m_pad, d, ctypes.c_float(ts), _ptr(q), _ptr(sf), rows)
    return q, sf


def sf_offset(r: int, c: int, cols: int) -> int:
    return int(lib().orc_sf_offset(r, c, cols))


def swizzle_sf(sf_logical: np.ndarray) -> np.ndarray:
    """Logical [rows, cols] scales -> the GEMM's 128x4-atom layout (flat bytes)."""
    sf = np.ascontiguousarray(sf_logical, dtype=np.uint8)
    rows, cols = sf.shape
    assert rows % 128 == 0 and cols % 4 == 0
    out = np.empty(rows * cols, dtype=np.uint8)
    lib().orc_swizzle_sf(_ptr(sf), rows, cols, _ptr(out))
    return out


def unswizzle_sf(flat: np.ndarray, rows: int, cols: int) -> np.ndarray:
    flat = np.ascontiguousarray(flat, dtype=np.uint8).reshape(-1)
    assert flat.size == rows * cols
    out = np.empty((rows, cols), dtype=np.uint8)
    lib().orc_unswizzle_sf(_ptr(flat), rows, cols, _ptr(out))
    return out


def modulate_producer(x, shift, scale, seg_off, m_pad: int):
    """Both producer passes: returns (ts, qdata, sf_logical, y, amax_bits)."""
    y = modulate(x, shift, scale, seg_off)
    amax = absmax(y)
    ts = tensor_scale(amax)
    q, sf = pack(y, m_pad, ts)
    return ts, q, sf, y, amax


def plain_producer(x, m_pad: int):
    """Both producer passes on an activation taken as it is (no fused transform):
    returns (ts, qdata, sf_logical, amax_bits)."""
    xs = _u16(x)
    amax = absmax(xs)
    ts = tensor_scale(amax)
    q, sf = pack(xs, m_pad, ts)
    return ts, q, sf, amax


# ----------------------------------------------------------------------------
# SwiGLU
# ----------------------------------------------------------------------------
def _round_fraction_bf16(q: Fraction, negative: bool) -> int:
    """bf16 pattern nearest to the exact rational |q| (ties to even), sign given."""
    a = abs(q)
    sign = 0x8000 if negative else 0
    if a == 0:
        return sign
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    E = max(e, -126)
    quantum = Fraction(2) ** (E - 7)
    r = round(a / quantum)        # Python rounds Fractions half to even
    res = r * quantum
    if res > Fraction(255) * Fraction(2) ** 120:
        return sign | 0x7F80
    f = struct.unpack("<I", struct.pack("<f", float(res)))[0]   # exact: res is a bf16 value
    return sign | (f >> 16)


def _silu_bf16_of(bits: int) -> int:
    g = bf16_value(bits)
    if g != g:
        return 0x7FC0
    if g == 0.0:
        return bits                      # silu(+-0) = +-0
    if g > 100.0:
        # g - silu(g) = g e^-g / (1 + e^-g) < 100 e^-100, far below half a bf16 ulp of g.
        return bits
    if g < -100.0:
        # |silu(g)| < |g| e^g <= 100 e^-100 < 2^-134 (half the smallest bf16 subnormal).
        return 0x8000
    with localcontext() as ctx:
        ctx.prec = 60
        d = Decimal(g)                   # exact: g is a binary float
        s = d / (1 + (-d).exp())
    return _round_fraction_bf16(Fraction(s), s < 0)


@functools.lru_cache(maxsize=None)
def silu_table() -> np.ndarray:
    """uint16[65536]: correctly rounded bf16 silu(g) = g / (1 + e^-g) per bf16 pattern g.

    The quotient is evaluated with 60 significant decimal digits and rounded
    exactly to bf16; a wrong rounding would need the true value to lie within
    about 1e-58 (relative) of a bf16 rounding boundary.
    """
    return np.array([_silu_bf16_of(b) for b in range(65536)], dtype=np.uint16)


def swiglu(gate, up) -> np.ndarray:
    g = _u16(gate)
    u = _u16(up)
    m, f = g.shape
    assert u.shape == (m, f)
    tab = silu_table()
    h = np.empty((m, f), dtype=np.uint16)
    lib().orc_swiglu(_ptr(g), f, _ptr(u), f, m, f, _ptr(tab), _ptr(h), f)
    return h


def swiglu_producer(gate, up, m_pad: int):
    """SwiGLU then both producer passes: returns (ts, qdata, sf_logical, h, amax_bits)."""
    h = swiglu(gate, up)
    amax = absmax(h)
    ts = tensor_scale(amax)
    q, sf = pack(h, m_pad, ts)
    return ts, q, sf, h, amax


# ----------------------------------------------------------------------------
# GEMM
# ----------------------------------------------------------------------------
def dequant(q, sf_logical, k: int, ts: float, r0: int = 0, r1: int | None = None) -> np.ndarray:
    """FP64 values e2m1(code) * e4m3(scale) * ts for rows [r0, r1)."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    sf = np.ascontiguousarray(sf_logical, dtype=np.uint8)
    if r1 is None:
        r1 = q.shape[0]
    assert q.shape[1] == k // 2 and sf.shape[1] == k // 16
    out = np.empty((r1 - r0, k), dtype=np.float64)
    lib().orc_dequant(_ptr(q), _ptr(sf), k, ctypes.c_float(ts), r0, r1, _ptr(out))
    return out


def gemm_reference(qa, sfa, ts_a, qb, sfb, ts_b, k: int, rows=None, n_chunk: int = 2048):
    """R[i, n] = sum_k a_k b_k and S[i, n] = sum_k |a_k b_k| in FP64.

    qa/sfa: activation codes [>=M, k/2] and logical scales; qb/sfb: weight
    codes [N, k/2] and logical scales [>=N, k/16].  rows: activation row
    indices to evaluate (default: all rows of qa).
    """
    qa = np.asarray(qa)
    if rows is None:
        rows = np.arange(qa.shape[0])
    rows = np.asarray(rows, dtype=np.int64)
    A = np.stack([dequant(qa, sfa, k, ts_a, int(r), int(r) + 1)[0] for r in rows]) if len(rows) else np.zeros((0, k))
    n = np.asarray(qb).shape[0]
    R = np.empty((len(rows), n), dtype=np.float64)
    S = np.empty((len(rows), n), dtype=np.float64)
    Aabs = np.abs(A)
    for n0 in range(0, n, n_chunk):
        n1 = min(n, n0 + n_chunk)
        B = dequant(qb, sfb, k, ts_b, n0, n1)
        R[:, n0:n1] = A @ B.T
        S[:, n0:n1] = Aabs @ np.abs(B).T
    return R, S


def gated_residual(c, gate, seg_off, res) -> np.ndarray:
    """out = RN_bf16(res + RN_bf16(gate_s * c)) per element, gate_s the gate row of
    the row's segment ("NVFP4 Streaming Design", P4).  c, res: uint16 [m, n];
    gate: uint16 [nseg, n]; seg_off: nseg + 1 row offsets (0 ... m)."""
    c, gate, res = _u16(c), _u16(gate), _u16(res)
    m, n = c.shape
    off = np.ascontiguousarray(np.asarray(seg_off, dtype=np.int32))
    nseg = len(off) - 1
    assert gate.shape == (nseg, n) and res.shape == (m, n)
    assert off[0] == 0 and off[-1] == m and np.all(np.diff(off) >= 0)
    out = np.empty((m, n), dtype=np.uint16)
    lib().orc_gated_residual(_ptr(c), n, _ptr(gate), n, _ptr(off), nseg, _ptr(res), n, m, n, _ptr(out), n)
    return out


def _bf16_directed(v: np.ndarray, up: bool) -> np.ndarray:
    """bf16 bit patterns of the smallest bf16 >= v (up) or the largest <= v,
    for finite v inside the bf16 range (no overflow handling needed here)."""
    v = np.asarray(v, dtype=np.float64)
    bits = np.array([bf16_bits(float(x)) for x in v.ravel()], dtype=np.int64).reshape(v.shape)
    vals = bf16_to_f64(bits.astype(np.uint16))
    need = (vals < v) if up else (vals > v)
    # one bf16 step in the needed direction: on the bit pattern, +1 moves away
    # from zero and -1 towards it; from +-0 the step goes to the smallest
    # subnormal of the needed sign
    pos, neg = vals > 0, vals < 0
    if up:
        step = np.where(pos, bits + 1, np.where(neg, bits - 1, 0x0001))
    else:
        step = np.where(pos, bits - 1, np.where(neg, bits + 1, 0x8001))
    return np.where(need, step, bits).astype(np.uint16)


def gated_residual_bounds(R, S, gate, seg_off, res):
    """Every output the gated epilogue may give for a GEMM result within the
    GEMM tolerance of R: with c ranging over the bf16 values in
    [R - tol, R + tol] (tol as in gemm_tolerance), out(c) = RN(res + RN(g c))
    is monotone in c (non-decreasing for g >= 0, non-increasing for g < 0), so
    the outputs lie between out(c_lo) and out(c_hi).  Returns (lo, hi) as
    float64 arrays."""
    tol = gemm_tolerance(R, S)
    c_lo = _bf16_directed(R - tol, up=True)
    c_hi = _bf16_directed(R + tol, up=False)
    o1 = bf16_to_f64(gated_residual(c_lo, gate, seg_off, res))
    o2 = bf16_to_f64(gated_residual(c_hi, gate, seg_off, res))
    return np.minimum(o1, o2), np.maximum(o1, o2)


def ulp_bf16(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |v| (2^-133 below the normal range and at 0)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -126.0)
    return np.where(a > 0, np.exp2(e - 7.0), 2.0 ** -133)


def gemm_tolerance(R: np.ndarray, S: np.ndarray) -> np.ndarray:
    """Allowed |C - R|: one bf16 ulp of R plus 1e-5 * sum_k |a_k b_k|."""
    return ulp_bf16(R) + 1e-5 * S


def gemm_check(C_bits: np.ndarray, R: np.ndarray, S: np.ndarray):
    """Returns (ok_mask, abs_err, tol) for bf16 output patterns C against R."""
    C = bf16_to_f64(_u16(C_bits))
    err = np.abs(C - R)
    tol = gemm_tolerance(R, S)
    return err <= tol, err, tol
