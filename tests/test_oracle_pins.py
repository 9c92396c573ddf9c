"""Pins of the CPU oracle against things other than itself (CPU only).

Each test checks one oracle function against brute force, a closed form, an
independent library routine (torch CPU bf16 arithmetic and float8 casts), or
hand-derived golden values, so that a dropped term, a wrong sign, a wrong
index or a transposed operand in the oracle fails at least one of them.
"""
import ctypes
import math
import os
import subprocess
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from dit_modulate_absmax_gb300 import workloads as W

HERE = os.path.dirname(os.path.abspath(__file__))


def _f32_bits_to_f64(u32):
    return np.asarray(u32, dtype=np.uint32).view(np.float32).astype(np.float64)


def _round_array(vals, p, emin, maxv, sat):
    L = oracle.lib()
    fn = L.orc_round_array
    fn.restype = None
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int,
                   ctypes.c_void_p]
    a = np.ascontiguousarray(vals, dtype=np.float64)
    out = np.empty_like(a)
    fn(a.ctypes.data, a.size, p, emin, maxv, sat, out.ctypes.data)
    return out


# ---------------------------------------------------------------------------
# Codecs
# ---------------------------------------------------------------------------
def test_codecs_exhaustive_vs_brute_force(tmp_path):
    """E2M1 and E4M3 encoders on every finite binary32 pattern vs nearest-value search."""
    exe = tmp_path / "codec_exhaustive"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-o", str(exe),
                           os.path.join(HERE, "helpers", "codec_exhaustive.c"), "-lm"])
    bad2, bad4, checked = map(int, subprocess.check_output([str(exe)], text=True).split())
    assert checked == 2 ** 32 - 2 * (2 ** 23 - 1)      # every pattern but the NaNs
    assert bad2 == 0 and bad4 == 0


def test_e4m3_decode_matches_torch_float8():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = oracle.e4m3_table()
    both_nan = np.isnan(ref) & np.isnan(mine)
    assert np.array_equal(np.isnan(ref), np.isnan(mine))
    assert np.array_equal(ref[~both_nan], mine[~both_nan])
    assert np.array_equal(np.signbit(ref[~both_nan]), np.signbit(mine[~both_nan]))


def test_e4m3_encode_matches_torch_float8_in_range():
    g = torch.Generator().manual_seed(11)
    v = torch.cat([
        (torch.rand(200_000, generator=g) * 2 - 1) * 448,
        (torch.rand(200_000, generator=g) * 2 - 1) * 2.0 ** -6,      # subnormal range
        torch.randn(200_000, generator=g),
    ]).to(torch.float32)
    ref = v.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    vd = v.to(torch.float64).numpy()
    L = oracle.lib()
    fn = L.orc_e4m3_encode_array
    fn.restype = None
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
    out = np.empty(vd.size, dtype=np.uint8)
    fn(vd.ctypes.data, vd.size, out.ctypes.data)
    assert np.array_equal(out, ref)


def test_e2m1_decode_from_bit_fields():
    # sign | 2 exponent bits (bias 1) | 1 mantissa bit; exponent 0 is subnormal (m * 0.5)
    for c in range(16):
        s, e, m = c >> 3, (c >> 1) & 3, c & 1
        mag = 0.5 * m if e == 0 else 2.0 ** (e - 1) * (1 + 0.5 * m)
        want = -mag if s else mag
        got = oracle.e2m1_decode(c)
        assert got == want and math.copysign(1, got) == math.copysign(1, want)


def test_e2m1_special_points():
    # midpoints go to the even code; saturation at 6; signed zero kept
    cases = [(0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6), (5.0001, 7), (1e30, 7),
             (-0.25, 8), (-0.0, 8), (0.0, 0), (-1e-40, 8), (float("inf"), 7), (float("-inf"), 15)]
    for v, c in cases:
        assert oracle.e2m1_encode(v) == c, v


# ---------------------------------------------------------------------------
# Rounding and modulation
# ---------------------------------------------------------------------------
def test_rn_bf16_matches_torch_conversion():
    g = torch.Generator().manual_seed(3)
    bits = torch.randint(0, 2 ** 31 - 1, (400_000,), generator=g, dtype=torch.int64)
    bits = torch.cat([bits, bits | 0x80000000, torch.arange(0, 2 ** 17) << 7])   # plus exact ties near zero
    u = bits.to(torch.int64).numpy().astype(np.uint32)
    f = torch.from_numpy(u.view(np.float32).copy())
    ok = torch.isfinite(f)
    f = f[ok]
    ref = f.to(torch.bfloat16).to(torch.float64).numpy()
    mine = _round_array(f.to(torch.float64).numpy(), 8, -126, float(np.ldexp(255.0, 120)), 0)
    fin = np.isfinite(ref)
    assert np.array_equal(np.isinf(ref), np.isinf(mine))
    assert np.array_equal(ref[fin], mine[fin])


def test_rn_f32_matches_numpy_float32_cast():
    rng = np.random.default_rng(4)
    v = np.concatenate([rng.standard_normal(100_000) * 10.0 ** rng.integers(-45, 38, 100_000),
                        rng.standard_normal(1000) * 1e-42])
    mine = _round_array(v, 24, -126, float(np.finfo(np.float32).max), 0)
    ref = v.astype(np.float32).astype(np.float64)      # IEEE round to nearest even
    assert np.array_equal(mine, ref)


def _torch_modulate(x, shift, scale):
    xb = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16)
    sh = torch.from_numpy(shift.view(np.int16).copy()).view(torch.bfloat16)
    sc = torch.from_numpy(scale.view(np.int16).copy()).view(torch.bfloat16)
    y = (xb * (sc + 1)) + sh          # three separately rounded bf16 ops
    return y.view(torch.int16).numpy().view(np.uint16)


def test_modulate_matches_torch_bf16_ops_random():
    rng = np.random.default_rng(5)
    m, d = 64, 256
    x = rng.integers(0, 65536, size=(m, d), dtype=np.uint16)
    x[(x & 0x7F80) == 0x7F80] = 0x3F80                 # keep inputs finite
    shift = (torch.randn(1, d) * 0.3).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    scale = (torch.randn(1, d) * 0.3).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    y = oracle.modulate(x, shift, scale, [0, m])
    ref = _torch_modulate(x, np.broadcast_to(shift, (m, d)).copy(), np.broadcast_to(scale, (m, d)).copy())
    nan = ((ref & 0x7FFF) > 0x7F80)
    assert np.array_equal(y[~nan], ref[~nan])
    assert np.array_equal((y & 0x7FFF) > 0x7F80, nan)


def test_modulate_exhaustive_x_matches_torch():
    """All 65,536 bf16 x against torch for a handful of (scale, shift) pairs."""
    xs = np.arange(65536, dtype=np.uint16).reshape(-1, 1)
    pairs = [(0.0, 0.0), (0.1, -0.2), (-0.37, 1.5), (3.0, -1e-38), (-1.0, 0.5), (1e-3, 2.0 ** -130)]
    for sc_v, sh_v in pairs:
        shift = np.array([[oracle.bf16_bits(sh_v)]], dtype=np.uint16)
        scale = np.array([[oracle.bf16_bits(sc_v)]], dtype=np.uint16)
        y = oracle.modulate(xs, shift, scale, [0, 65536])
        ref = _torch_modulate(xs, np.broadcast_to(shift, xs.shape).copy(), np.broadcast_to(scale, xs.shape).copy())
        nan = (ref & 0x7FFF) > 0x7F80
        assert np.array_equal(nan, (y & 0x7FFF) > 0x7F80)
        assert np.array_equal(y[~nan], ref[~nan]), (sc_v, sh_v)


def test_modulate_uses_each_rows_segment():
    rng = np.random.default_rng(6)
    m, d = 10, 256
    x = (torch.randn(m, d) ).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    shift = (torch.randn(3, d)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    scale = (torch.randn(3, d)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    off = [0, 4, 4, 10]                                # segment 1 is empty
    y = oracle.modulate(x, shift, scale, off)
    for r in range(m):
        s = 0 if r < 4 else 2
        ref = _torch_modulate(x[r:r + 1], shift[s:s + 1], scale[s:s + 1])
        assert np.array_equal(y[r:r + 1], ref)


# ---------------------------------------------------------------------------
# Absmax and tensor scale
# ---------------------------------------------------------------------------
def test_absmax_matches_numpy_and_is_order_free():
    rng = np.random.default_rng(7)
    y = (torch.randn(50, 256) * 3).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ref = np.abs(oracle.bf16_to_f64(y)).max()
    assert oracle.bf16_value(oracle.absmax(y)) == ref
    perm = y[rng.permutation(50)][:, rng.permutation(256)].copy()
    assert oracle.absmax(perm) == oracle.absmax(y)


def test_absmax_special_values():
    y = np.zeros((2, 16), dtype=np.uint16)
    y[0, 3] = 0x8000                                   # -0
    assert oracle.absmax(y) == 0
    y[1, 5] = 0xC080                                   # -4
    assert oracle.bf16_value(oracle.absmax(y)) == 4.0
    y[0, 0] = 0x7FC1                                   # NaN wins
    assert (oracle.absmax(y) & 0x7FFF) > 0x7F80


def test_tensor_scale_closed_forms():
    assert oracle.tensor_scale(oracle.bf16_bits(2688.0)) == 1.0
    assert oracle.tensor_scale(oracle.bf16_bits(10752.0)) == 4.0
    assert oracle.tensor_scale(0) == 0.0
    for v in (1.0, 3.140625, 1e-30, 3e38, 2.0 ** -133):
        want = float(np.float32(np.float32(oracle.rn_bf16(v)) / np.float32(2688.0)))
        assert oracle.tensor_scale(oracle.bf16_bits(v)) == want


# ---------------------------------------------------------------------------
# Pack
# ---------------------------------------------------------------------------
def _golden_blocks():
    rows = []
    with open(os.path.join(HERE, "golden", "pack_blocks.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            name, ts, ys, sfc, qb = [p.strip() for p in line.split("|")]
            rows.append((name, float(ts), [float(v) for v in ys.split()], int(sfc, 16),
                         [int(b, 16) for b in qb.split()]))
    return rows


@pytest.mark.parametrize("block", _golden_blocks(), ids=lambda b: b[0])
def test_pack_golden_blocks(block):
    name, ts, ys, sfc, qb = block
    assert len(ys) == 16 and len(qb) == 8
    y = np.array([[oracle.bf16_bits(v) if not (v == 0 and math.copysign(1, v) < 0) else 0x8000 for v in ys]],
                 dtype=np.uint16)
    for v, b in zip(ys, y[0]):
        assert oracle.bf16_value(b) == v           # inputs are exact bf16 values
    q, sf = oracle.pack(y, 16, ts)
    assert sf[0, 0] == sfc, (name, hex(sf[0, 0]))
    assert list(q[0]) == qb, (name, [hex(v) for v in q[0]])
    assert not q[1:].any() and not sf[1:].any()


def _nearest_e2m1_codes(qv):
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    a = np.minimum(np.abs(qv), 6.0)
    dist = np.abs(a[..., None] - mags)
    best = dist.min(-1, keepdims=True)
    cand = dist == best
    # among equidistant codes prefer the even one
    idx = np.where(cand[..., ::2].any(-1), np.argmax(cand & (np.arange(8) % 2 == 0), -1), np.argmax(cand, -1))
    return idx | np.where(np.signbit(qv), 8, 0)


def test_pack_tiny_adversarial_properties():
    """Every code and scale of the adversarial tiny case is the nearest representable value."""
    from oracle.adversarial import tiny_adversarial
    w = W.WORKLOADS["tiny"]
    a = W.activations(w)
    off = W.seg_offsets(w)
    sh = a["shift"].numpy().view(np.uint16)
    sc = a["scale"].numpy().view(np.uint16)
    x = tiny_adversarial(a["x"].numpy().view(np.uint16), sh, sc, off)
    ts, q, sf, y, amax = oracle.modulate_producer(x, sh, sc, off, w.m_pad)
    assert ts == 4.0 and oracle.bf16_value(amax) == 10752.0
    yv = oracle.bf16_to_f64(y).reshape(w.m, -1, 16)
    bamax = np.abs(yv).max(-1)
    den = np.float32(6.0) * np.float32(ts)
    ratio = (bamax.astype(np.float32) / den).astype(np.float32)
    want_sf = torch.from_numpy(ratio).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    want_sf[bamax == 0] = 0
    assert np.array_equal(sf[: w.m], want_sf)
    scv = (oracle.e4m3_table()[sf[: w.m]].astype(np.float32) * np.float32(ts)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        qv = (yv.astype(np.float32) / scv[..., None]).astype(np.float32).astype(np.float64)
    codes = np.where(scv[..., None] == 0, np.where(np.signbit(yv), 8, 0), _nearest_e2m1_codes(qv))
    lo = q[: w.m].reshape(w.m, -1, 8) & 0xF
    hi = q[: w.m].reshape(w.m, -1, 8) >> 4
    got = np.stack([lo, hi], -1).reshape(w.m, -1, 16)
    assert np.array_equal(got, codes)
    assert not q[w.m:].any() and not sf[w.m:].any()
    # the adversarial rows really exercise what they should
    mid = np.isin(np.abs(qv[[10, 11, 12, 13, 260, 261]]), [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]).sum()
    assert mid > 1000
    assert (sf[[20, 21, 270]] == 0).sum() >= 4                 # all-zero blocks
    assert ((sf[[30, 31, 280]] < 8) & (sf[[30, 31, 280]] > 0)).sum() >= 8   # subnormal scales
    assert (sf[[30, 31, 280]] == 0).sum() >= 4                 # scales that round to zero


def _codes(q, m):
    lo, hi = q[:m] & 0xF, q[:m] >> 4
    return np.stack([lo, hi], -1).reshape(m, -1)


def test_pack_non_finite_inputs_hand_derived():
    """NaN and infinity, by hand from the formulas in IEEE arithmetic and the
    two stated conventions (a NaN quotient is the E4M3 NaN code 0x7F; a zero
    or NaN scale product gives zeros with y's signs).

    NaN tensor: amax and ts are NaN, so every block with a nonzero maximum has
    quotient NaN -> 0x7F and an all-zero block keeps 0; every scale product
    (NaN * anything, 0 * NaN) is NaN, so every code is a signed zero.
    Infinite tensor: ts = RN(inf / 2688) = inf; the block holding the infinity
    has quotient inf / inf = NaN -> 0x7F, a finite nonzero block has
    quotient 0 -> 0, and every scale product (NaN * inf, 0 * inf) is NaN."""
    nan, pinf, neg_zero = 0x7FC0, 0x7F80, 0x8000
    one, two, mthree = 0x3F80, 0x4000, 0xC040
    y = np.zeros((2, 64), dtype=np.uint16)
    y[0, 0:16] = one
    y[0, 3] = nan                        # block 0: NaN among finite values
    y[0, 16:32] = 0
    y[0, 20] = neg_zero                  # block 1: all zero (one -0)
    y[0, 32:48] = mthree                 # block 2: finite, negative
    y[0, 48:64] = nan | 0x8000           # block 3: negative NaNs only
    y[1, :] = two
    ts = oracle.tensor_scale(oracle.absmax(y))
    assert np.isnan(ts)
    q, sf = oracle.pack(y, 16, ts)
    assert sf[0].tolist() == [0x7F, 0x00, 0x7F, 0x7F] and sf[1].tolist() == [0x7F] * 4
    want = np.where(y.view(np.int16) < 0, 8, 0)      # zeros with y's signs
    assert np.array_equal(_codes(q, 2), want)
    assert not q[2:].any() and not sf[2:].any()

    y = np.zeros((1, 48), dtype=np.uint16)
    y[0, 0:16] = one
    y[0, 5] = pinf                       # block 0 holds +inf
    y[0, 16:32] = mthree                 # block 1 finite
    y[0, 40] = neg_zero                  # block 2 all zero
    ts = oracle.tensor_scale(oracle.absmax(y))
    assert ts == float("inf")
    q, sf = oracle.pack(y, 16, ts)
    assert sf[0].tolist() == [0x7F, 0x00, 0x00]
    assert np.array_equal(_codes(q, 1), np.where(y.view(np.int16) < 0, 8, 0))


# ---------------------------------------------------------------------------
# Scale layout
# ---------------------------------------------------------------------------
def test_sf_layout_atoms_and_bijection():
    rows, cols = 256, 32
    # facts of the 128x4-atom layout: 16 bytes per row of 32, 4 bytes per 32-row group
    assert oracle.sf_offset(0, 0, cols) == 0
    assert oracle.sf_offset(1, 0, cols) == 16
    assert oracle.sf_offset(32, 0, cols) == 4
    assert oracle.sf_offset(0, 1, cols) == 1
    assert oracle.sf_offset(0, 4, cols) == 512
    assert oracle.sf_offset(128, 0, cols) == 512 * (cols // 4)
    offs = {oracle.sf_offset(r, c, cols) for r in range(rows) for c in range(cols)}
    assert offs == set(range(rows * cols))
    rng = np.random.default_rng(8)
    sf = rng.integers(0, 256, size=(rows, cols), dtype=np.uint8)
    assert np.array_equal(oracle.unswizzle_sf(oracle.swizzle_sf(sf), rows, cols), sf)


# ---------------------------------------------------------------------------
# SwiGLU
# ---------------------------------------------------------------------------
def _bits_to_float(b):
    return float(np.uint32(int(b) << 16).view(np.float32))


def test_silu_table_special_values_and_limits():
    tab = oracle.silu_table()
    assert tab[0x0000] == 0x0000 and tab[0x8000] == 0x8000
    for v in (8.0, 9.0, 100.0, 1e10, 3e38):
        b = oracle.bf16_bits(v)
        assert tab[b] == b                                  # silu(g) rounds to g for g >= 8
    for v in (-200.0, -1e10):
        assert tab[oracle.bf16_bits(v)] == 0x8000           # underflows to -0
    assert tab[0x7F80] == 0x7F80
    # global minimum of silu is about -0.2785 at g = -1.2785
    finite = [b for b in range(65536) if (b & 0x7F80) != 0x7F80]
    vals = np.array([_bits_to_float(tab[b]) for b in finite])
    assert vals.min() == -0.279296875          # bf16 nearest to the true minimum -0.27846


def test_silu_table_agrees_with_double_evaluation():
    """Away from bf16 rounding boundaries, rounding a double evaluation must agree."""
    tab = oracle.silu_table()
    n_checked = 0
    for b in range(65536):
        if (b & 0x7F80) == 0x7F80:
            continue
        g = _bits_to_float(b)
        if g < -100 or g > 100 or g == 0:
            continue
        v = g / (1.0 + math.exp(-g))
        f = np.float32(v)
        # skip values whose double evaluation sits within 1e-9 (relative) of a bf16 rounding boundary
        u = int(f.view(np.uint32))
        up = np.uint32(((u >> 16) << 16) + 0x8000).view(np.float32)
        if abs(float(up) - v) <= 1e-9 * abs(v):
            continue
        want = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
        assert tab[b] == want, (hex(b), g)
        n_checked += 1
    assert n_checked > 30000                 # every bf16 pattern with 0 < |g| <= 100, less near-ties


def test_silu_identity_silu_g_minus_silu_neg_g_is_g():
    tab = oracle.silu_table()
    rng = np.random.default_rng(9)
    for b in rng.integers(0, 0x7F80, size=2000):
        g = _bits_to_float(b)
        a = _bits_to_float(tab[b])
        c = _bits_to_float(tab[b | 0x8000])
        # each side is within half a bf16 ulp of the exact value
        tol = 2.0 ** (math.floor(math.log2(max(abs(a), 2.0 ** -126))) - 8) + 2.0 ** (
            math.floor(math.log2(max(abs(c), 2.0 ** -126))) - 8) + 2.0 ** -133
        assert abs((a - c) - g) <= tol * 1.0000001, (hex(b), g, a, c)


def test_swiglu_is_rounded_product():
    g = (torch.randn(8, 256) * 3).to(torch.bfloat16)
    u = torch.randn(8, 256).to(torch.bfloat16)
    h = oracle.swiglu(g.view(torch.int16).numpy(), u.view(torch.int16).numpy())
    tab = oracle.silu_table()
    sg = torch.from_numpy(tab[g.view(torch.int16).numpy().view(np.uint16)].view(np.int16)).view(torch.bfloat16)
    ref = (sg * u).view(torch.int16).numpy().view(np.uint16)      # torch bf16 multiply
    assert np.array_equal(h, ref)


def test_plain_producer_is_identity_modulation_except_negative_zero():
    """Without a fused transform the producer packs x itself.  With shift = scale
    = 0 the modulation is y = RN(RN(x * RN(0 + 1)) + 0) = x wherever x is not -0,
    so both producers must give the same bytes there (the modulation producer is
    pinned to torch's bf16 arithmetic above); at x = -0 the modulation's +0
    shift gives +0 (E2M1 code 0x0) while the plain producer keeps the sign
    (code 0x8)."""
    g = torch.Generator().manual_seed(41)
    x = (torch.randn(130, 512, generator=g) * 3).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
    x[x == 0x8000] = 0
    zero = np.zeros((1, 512), dtype=np.uint16)
    ts_p, q_p, sf_p, _ = oracle.plain_producer(x, 144)
    ts_m, q_m, sf_m, _, _ = oracle.modulate_producer(x, zero, zero, [0, 130], 144)
    assert ts_p == ts_m and np.array_equal(q_p, q_m) and np.array_equal(sf_p, sf_m)
    x[5, 17] = 0x8000                       # element 17: high nibble of byte 8 of row 5
    _, q_p, _, _ = oracle.plain_producer(x, 144)
    _, q_m, _, _, _ = oracle.modulate_producer(x, zero, zero, [0, 130], 144)
    assert q_p[5, 8] >> 4 == 0x8 and q_m[5, 8] >> 4 == 0x0
    assert np.array_equal(np.delete(q_p.ravel(), 5 * 256 + 8), np.delete(q_m.ravel(), 5 * 256 + 8))


def test_gated_residual_matches_torch_bf16_ops():
    """out = RN(res + RN(gate_s * c)): torch's CPU bf16 tensors round every
    elementwise operation, so `res + gate * c` in bf16 is the same sequence."""
    g = torch.Generator().manual_seed(43)
    c = (torch.randn(7, 256, generator=g) * 50).to(torch.bfloat16)
    gate = torch.randn(3, 256, generator=g).to(torch.bfloat16)
    res = (torch.randn(7, 256, generator=g) * 20).to(torch.bfloat16)
    c[0, :4] = torch.tensor([0.0, -0.0, 1e-38, -3e38])
    gate[0, :4] = torch.tensor([-0.0, 2.0, 1e-3, 0.5])
    res[0, :4] = torch.tensor([-0.0, -0.0, 1e38, 3e38])
    off = [0, 2, 2, 7]                      # an empty middle segment
    bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)
    out = oracle.gated_residual(bits(c), bits(gate), off, bits(res))
    gsel = torch.cat([gate[0:1].expand(2, 256), gate[2:3].expand(5, 256)])
    assert np.array_equal(out, bits(res + gsel * c))


def _all_finite_bf16():
    """Every finite bf16 value, sorted (from the 2^16 patterns through torch's bf16 view)."""
    pats = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).double().numpy()
    return np.unique(pats[np.isfinite(pats)])


def test_bf16_directed_rounding_matches_brute_force():
    """_bf16_directed(v, up) is the smallest bf16 >= v (up) or the largest <= v,
    found here by binary search over the sorted list of every finite bf16."""
    allv = _all_finite_bf16()
    rng = np.random.default_rng(47)
    v = np.concatenate([
        rng.standard_normal(2000) * 10.0 ** rng.integers(-40, 38, size=2000),
        allv[rng.integers(0, allv.size, size=500)],                       # exact bf16 values
        (allv[1000:1500] + allv[1001:1501]) / 2,                          # exact midpoints
        [0.0, -0.0, 1e-45, -1e-45, 2.0 ** -133, -(2.0 ** -133), 2.0 ** -126, 3.0e38, -3.0e38],
    ])
    v = v[np.abs(v) <= allv[-1]]
    up = oracle.bf16_to_f64(oracle._bf16_directed(v, up=True))
    down = oracle.bf16_to_f64(oracle._bf16_directed(v, up=False))
    want_up = allv[np.searchsorted(allv, v, side="left")]
    want_down = allv[np.searchsorted(allv, v, side="right") - 1]
    assert np.array_equal(up, want_up)
    assert np.array_equal(down, want_down)


def test_gated_residual_bounds_match_brute_force_over_the_tolerance_interval():
    """gated_residual_bounds(R, S, ...) returns the smallest and largest output of
    the gated epilogue over every bf16 value c within the GEMM tolerance of R:
    enumerate those c one by one and evaluate RN(res + RN(gate_s * c)) with
    torch's CPU bf16 ops (an independent evaluator), then compare."""
    allv = _all_finite_bf16()
    rng = np.random.default_rng(53)
    m, n = 6, 24
    R = rng.standard_normal((m, n)) * 4.0
    R[0, :4] = [0.0, 1e-3, -1e-3, 5e-39]                  # intervals that contain or reach 0
    S = np.abs(R) * rng.uniform(1.0, 400.0, size=(m, n)) + 1e-3
    gate_t = torch.randn(2, n, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    gate_t[1, :6] = torch.tensor([-2.0, -0.5, 0.0, -0.0, 3.0, -1e-3])  # negative gates: decreasing maps
    res_t = (torch.randn(m, n, generator=torch.Generator().manual_seed(4)) * 8).to(torch.bfloat16)
    off = [0, 3, m]
    bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)
    lo, hi = oracle.gated_residual_bounds(R, S, bits(gate_t), off, bits(res_t))
    tol = oracle.gemm_tolerance(R, S)
    counted = 0
    for i in range(m):
        g = gate_t[0 if i < 3 else 1]
        for j in range(n):
            cs = allv[(allv >= R[i, j] - tol[i, j]) & (allv <= R[i, j] + tol[i, j])]
            assert cs.size >= 1
            counted += cs.size
            c = torch.tensor(cs, dtype=torch.float64).to(torch.bfloat16)
            outs = (res_t[i, j] + g[j] * c).double().numpy()
            assert lo[i, j] == outs.min() and hi[i, j] == outs.max(), (i, j, cs.size)
    assert counted > 10 * m * n   # the intervals hold many candidates, not just R's neighbours


# ---------------------------------------------------------------------------
# GEMM reference
# ---------------------------------------------------------------------------
def _exact_sum(qa_row, sfa_row, ts_a, qb_row, sfb_row, ts_b, k):
    def dec(q, sf, j):
        byte = int(q[j // 2])
        code = (byte >> 4) if j & 1 else (byte & 0xF)
        e, m, s = (code >> 1) & 3, code & 1, code >> 3
        mag = Fraction(m, 2) if e == 0 else Fraction(2) ** (e - 1) * (1 + Fraction(m, 2))
        c = int(sf[j // 16])
        ee, mm = (c >> 3) & 15, c & 7
        smag = Fraction(mm, 512) if ee == 0 else Fraction(2) ** (ee - 7) * (1 + Fraction(mm, 8))
        return (-mag if s else mag) * smag
    tot = Fraction(0)
    absum = Fraction(0)
    for j in range(k):
        p = dec(qa_row, sfa_row, j) * dec(qb_row, sfb_row, j)
        tot += p
        absum += abs(p)
    return tot * Fraction(ts_a) * Fraction(ts_b), absum * abs(Fraction(ts_a) * Fraction(ts_b))


def test_gemm_reference_matches_exact_rational_sums():
    rng = np.random.default_rng(10)
    m, n, k = 3, 5, 64
    qa = rng.integers(0, 256, size=(m, k // 2), dtype=np.uint8)
    qb = rng.integers(0, 256, size=(n, k // 2), dtype=np.uint8)
    sfa = np.zeros((128, k // 16), dtype=np.uint8)
    sfb = np.zeros((128, k // 16), dtype=np.uint8)
    sfa[:m] = rng.integers(0x20, 0x60, size=(m, k // 16))
    sfb[:n] = rng.integers(0x01, 0x60, size=(n, k // 16))
    ts_a, ts_b = 0.375, 2.0 ** -10
    R, S = oracle.gemm_reference(qa, sfa, ts_a, qb, sfb, ts_b, k)
    for i in range(m):
        for j in range(n):
            tot, absum = _exact_sum(qa[i], sfa[i], ts_a, qb[j], sfb[j], ts_b, k)
            assert R[i, j] == float(tot)          # exact: every partial sum is representable
            assert S[i, j] == float(absum)


def test_gemm_reference_is_not_transposed():
    # one nonzero code per operand: C[i, j] is nonzero only where both rows meet
    k = 32
    qa = np.zeros((2, k // 2), dtype=np.uint8)
    qb = np.zeros((3, k // 2), dtype=np.uint8)
    qa[1, 0] = 0x02          # a[1, 0] = 1.0
    qb[2, 0] = 0x07          # b[2, 0] = 6.0
    sfa = np.full((128, 2), 0x38, dtype=np.uint8)
    sfb = np.full((128, 2), 0x38, dtype=np.uint8)
    R, S = oracle.gemm_reference(qa, sfa, 1.0, qb, sfb, 1.0, k)
    want = np.zeros((2, 3))
    want[1, 2] = 6.0
    assert np.array_equal(R, want) and np.array_equal(S, want)


def test_ulp_bf16_and_tolerance():
    assert oracle.ulp_bf16(np.array([1.0]))[0] == 2.0 ** -7
    assert oracle.ulp_bf16(np.array([1.99]))[0] == 2.0 ** -7
    assert oracle.ulp_bf16(np.array([-2.0]))[0] == 2.0 ** -6
    assert oracle.ulp_bf16(np.array([2.0 ** -130]))[0] == 2.0 ** -133
    assert oracle.ulp_bf16(np.array([0.0]))[0] == 2.0 ** -133
    R = np.array([[1.0]])
    S = np.array([[1000.0]])
    ok, _, tol = oracle.gemm_check(np.array([[oracle.bf16_bits(1.0078125)]], dtype=np.uint16), R, S)
    assert ok.all() and tol[0, 0] == 2.0 ** -7 + 1e-2
