"""GPU parity of the two-pass NVFP4 producers against the CPU oracle.

The tensor scale, every QDATA byte and every scale byte (compared after the
oracle applies its own scale layout) must match bit for bit.  Output buffers
are pre-filled with a canary so that a byte the kernels fail to write shows.
"""
import numpy as np
import pytest
import torch

import oracle
from dit_modulate_absmax_gb300 import workloads as W

pytestmark = pytest.mark.gpu
CANARY = 0xAB


def _u16(t):
    return t.cpu().numpy().view(np.uint16)


def _to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def _f32_bits(v):
    return int(np.float32(v).view(np.uint32))


def run_modulate(h3, x, sh, sc, off, m_pad, x_dev=None):
    m, d = x.shape
    xd = _to_dev(x) if x_dev is None else x_dev
    shd, scd = _to_dev(sh), _to_dev(sc)
    q = torch.full((m_pad, d // 2), CANARY, dtype=torch.uint8, device="cuda")
    sfa = torch.full((h3.sf_bytes(m_pad, d),), CANARY, dtype=torch.uint8, device="cuda")
    ts = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
    h3.modulate_absmax(xd, shd, scd, off, tensor_scale=ts)
    h3.modulate_pack(xd, shd, scd, off, ts, m_pad, qdata=q, sfa=sfa)
    torch.cuda.synchronize()
    assert h3.h3fp4_device_error() == 0
    return float(ts.item()), q.cpu().numpy(), sfa.cpu().numpy()


def check_modulate(h3, x, sh, sc, off, m_pad):
    ts_o, q_o, sf_o, _, _ = oracle.modulate_producer(x, sh, sc, off, m_pad)
    ts, q, sfa = run_modulate(h3, x, sh, sc, off, m_pad)
    assert _f32_bits(ts) == _f32_bits(ts_o), (ts, ts_o)
    assert np.array_equal(q, q_o), f"QDATA differs at {np.argwhere(q != q_o)[:5].tolist()}"
    want = oracle.swizzle_sf(sf_o)
    assert np.array_equal(sfa, want), f"SFA differs at {np.argwhere(sfa != want)[:5].tolist()}"
    return ts


def _bf16(t):
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _random_case(m, d, nseg, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    x = _bf16(torch.randn(m, d, generator=g) * scale)
    sh = _bf16(torch.randn(nseg, d, generator=g) * 0.2)
    sc = _bf16(torch.randn(nseg, d, generator=g) * 0.2)
    return x, sh, sc


def test_tiny_adversarial_bit_exact(h3):
    from oracle.adversarial import tiny_adversarial
    w = W.WORKLOADS["tiny"]
    a = W.activations(w)
    off = W.seg_offsets(w)
    sh = a["shift"].numpy().view(np.uint16)
    sc = a["scale"].numpy().view(np.uint16)
    x = tiny_adversarial(a["x"].numpy().view(np.uint16), sh, sc, off)
    ts = check_modulate(h3, x, sh, sc, off, w.m_pad)
    assert ts == 4.0


def test_tiny_plain_bit_exact(h3):
    w = W.WORKLOADS["tiny"]
    a = W.activations(w)
    check_modulate(h3, _u16(a["x"]), _u16(a["shift"]), _u16(a["scale"]), W.seg_offsets(w), w.m_pad)


@pytest.mark.parametrize("m,m_pad,d,off", [
    (1, 16, 256, [0, 1]),
    (129, 144, 512, [0, 100, 129]),
    (300, 320, 768, [0, 0, 150, 300]),            # empty first segment
    (1000, 1024, 256, [0, 200, 200, 700, 1000]),  # empty middle segment
    (257, 384, 256, [0, 257]),                    # m_pad well past m
    (640, 640, 1024, [0, 128, 256, 384, 512, 640]),
])
def test_ragged_shapes_bit_exact(h3, m, m_pad, d, off):
    x, sh, sc = _random_case(m, d, len(off) - 1, seed=m + d)
    check_modulate(h3, x, sh, sc, off, m_pad)


def test_ctas_walking_several_tiles_bit_exact(h3):
    """Pass 1 runs a capped persistent grid: at this size every CTA walks several
    tiles in different column slabs, with the largest |y| in a late tile."""
    m, d = 16384 + 77, 4096                    # 129 x 16 = 2064 tiles, more than the grid
    x, sh, sc = _random_case(m, d, 2, seed=18)
    x[16300, 3000] = oracle.bf16_bits(900.0)   # the global maximum, far from the first tiles
    check_modulate(h3, x, sh, sc, [0, 9000, m], m + 3)


def test_many_blocks_bit_exact(h3):
    """16.8 M values: enough quotients land within a few ulps of an E2M1 or E4M3
    rounding boundary to exercise both sides of the reciprocal fast path."""
    m, d = 8192, 2048
    x, sh, sc = _random_case(m, d, 2, seed=19, scale=3.0)
    check_modulate(h3, x, sh, sc, [0, 5000, m], m)


def test_many_segments_bit_exact(h3):
    m, d = 700, 256
    off = list(range(0, 700, 50)) + [700]          # 14 segments of 50 rows
    x, sh, sc = _random_case(m, d, len(off) - 1, seed=21)
    check_modulate(h3, x, sh, sc, off, 704)


def test_wide_dynamic_range_and_subnormals(h3):
    rng = np.random.default_rng(12)
    m, d = 200, 512
    mag = 10.0 ** rng.uniform(-40, 30, size=(m, d))
    x = _bf16(torch.from_numpy(mag * rng.choice([-1.0, 1.0], size=(m, d))).float())
    x[5] = rng.integers(1, 0x80, size=d).astype(np.uint16)            # subnormal x
    x[6] = x[5] | 0x8000
    x[7] = 0x8000                                                       # -0 row
    sh = _bf16(torch.randn(1, d) * 1e-20)
    sc = _bf16(torch.randn(1, d) * 0.5)
    check_modulate(h3, x, sh, sc, [0, m], 208)


def test_small_amax_tensor(h3):
    # every value tiny: tensor scale in the fp32 subnormal range, block scales saturate or vanish
    m, d = 64, 256
    x, sh, sc = _random_case(m, d, 1, seed=13, scale=1e-36)
    sh[:] = 0
    check_modulate(h3, x, sh, sc, [0, m], 64)


@pytest.mark.parametrize("log2_amax", [-60, -78, -79, -80, -81, -84, 100, 107, 108, 109, 110, 127])
def test_tensor_scales_at_the_edges_of_the_division_free_range(h3, log2_amax):
    """The pack divides without a division instruction while 6 ts lies in
    [2^-88, 2^100] and a block's scale product in [2^-100, 2^100], and by the
    IEEE division outside; tensors whose absolute maximum puts 6 ts on either
    side of those limits, with rows spanning 30 binades (so that block scale
    products fall on both sides too), must still match the oracle bit for bit."""
    m, d = 120, 512
    g = torch.Generator().manual_seed(40 + log2_amax)
    rows = torch.pow(2.0, -0.25 * torch.arange(m, dtype=torch.float64)).unsqueeze(1)
    v = torch.randn(m, d, generator=g, dtype=torch.float64) * rows
    v = v / v.abs().max() * 2.0 ** log2_amax
    x = _bf16(v.float())
    sh = np.zeros((1, d), dtype=np.uint16)
    sc = _bf16(torch.randn(1, d, generator=g) * 0.01)
    check_modulate(h3, x, sh, sc, [0, m], 128)


def test_zero_rows_gives_zero_scale(h3):
    d, m_pad = 256, 32
    x = np.zeros((0, d), dtype=np.uint16)
    sh = np.zeros((1, d), dtype=np.uint16)
    xd = torch.zeros((1, d), dtype=torch.int16, device="cuda")[:0]
    ts, q, sfa = run_modulate(h3, x, sh, sh, [0, 0], m_pad, x_dev=xd)
    assert ts == 0.0 and not q.any() and not sfa.any()


def test_all_zero_tensor(h3):
    m, d = 50, 256
    x = np.zeros((m, d), dtype=np.uint16)
    x[3, 7] = 0x8000
    sh = np.zeros((1, d), dtype=np.uint16)
    ts = check_modulate(h3, x, sh, sh, [0, m], 64)
    assert ts == 0.0


def _same_scale(ts, ts_o):
    """Equal tensor scales: the same bits, or both NaN (the payload is not specified)."""
    return (np.isnan(ts) and np.isnan(ts_o)) or _f32_bits(ts) == _f32_bits(ts_o)


NON_FINITE = {"nan": 0x7FC0, "neg_nan": 0xFFC0, "inf": 0x7F80, "neg_inf": 0xFF80}


@pytest.mark.parametrize("kind", list(NON_FINITE))
def test_non_finite_inputs_bit_exact(h3, kind):
    """A NaN or an infinity in the input: the tensor scale is NaN or infinite and
    the oracle's stated conventions decide the bytes (a NaN quotient is the
    E4M3 NaN code 0x7F, a zero or NaN scale product gives signed zeros); the
    modulation producer, the plain producer and the SwiGLU producer (with and
    without the h workspace) must match them byte for byte."""
    v = NON_FINITE[kind]
    m, d = 40, 512
    x, sh, sc = _random_case(m, d, 1, seed=14)
    sh[:] = 0                                # keep the planted value through the modulation
    x[4, 9] = v
    x[7, 16:32] = 0                          # an all-zero block
    x[7, 40] = 0x8000
    x[11, 64:80] = v                         # a block of nothing but the planted value
    ts_o, q_o, sf_o, _, _ = oracle.modulate_producer(x, sh, sc, [0, m], 48)
    ts, q, sfa = run_modulate(h3, x, sh, sc, [0, m], 48)
    assert np.isnan(ts_o) if "nan" in kind else np.isinf(ts_o)
    assert _same_scale(ts, ts_o), (ts, ts_o)
    assert np.array_equal(q, q_o), f"QDATA differs at {np.argwhere(q != q_o)[:5].tolist()}"
    assert np.array_equal(sfa, oracle.swizzle_sf(sf_o))
    assert (sf_o[:m] == 0x7F).any() and not q_o[:m][q_o[:m] & 0x77 != 0].any()

    ts_o, q_o, sf_o, _ = oracle.plain_producer(x, 48)
    ts, q, sfa = run_plain(h3, x, 48)
    assert _same_scale(ts, ts_o) and np.array_equal(q, q_o) and np.array_equal(sfa, oracle.swizzle_sf(sf_o))

    g = _bf16(torch.randn(m, d, generator=torch.Generator().manual_seed(15)))
    u = x.copy()                             # h = silu(g) * u carries the planted value
    ts_o, q_o, sf_o, h_o, _ = oracle.swiglu_producer(g, u, 48)
    for workspace in (False, True):
        ts, q, sfa, h = run_swiglu(h3, g, u, 48, workspace)
        assert _same_scale(ts, ts_o), (workspace, ts, ts_o)
        assert np.array_equal(q, q_o) and np.array_equal(sfa, oracle.swizzle_sf(sf_o)), workspace


def test_leading_dimensions(h3):
    m, d, ldx, ldm = 100, 256, 384, 264
    g = torch.Generator().manual_seed(15)
    xw = torch.randn(m, ldx, generator=g).to(torch.bfloat16).view(torch.int16)
    shw = (torch.randn(2, ldm, generator=g) * 0.2).to(torch.bfloat16).view(torch.int16)
    scw = (torch.randn(2, ldm, generator=g) * 0.2).to(torch.bfloat16).view(torch.int16)
    off = [0, 60, 100]
    ts_o, q_o, sf_o, _, _ = oracle.modulate_producer(_u16(xw[:, :d].contiguous()), _u16(shw[:, :d].contiguous()),
                                                     _u16(scw[:, :d].contiguous()), off, 112)
    xd, shd, scd = xw.cuda()[:, :d], shw.cuda()[:, :d], scw.cuda()[:, :d]
    ts = h3.modulate_absmax(xd, shd, scd, off)
    q, sfa = h3.modulate_pack(xd, shd, scd, off, ts, 112)
    torch.cuda.synchronize()
    assert float(ts.item()) == ts_o
    assert np.array_equal(q.cpu().numpy(), q_o)
    assert np.array_equal(sfa.cpu().numpy(), oracle.swizzle_sf(sf_o))


def test_repeated_calls_are_deterministic(h3):
    x, sh, sc = _random_case(500, 512, 2, seed=16)
    a = run_modulate(h3, x, sh, sc, [0, 300, 500], 512)
    b = run_modulate(h3, x, sh, sc, [0, 300, 500], 512)
    assert a[0] == b[0] and np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])


# ---------------------------------------------------------------------------
# SwiGLU producer
# ---------------------------------------------------------------------------
def run_swiglu(h3, g, u, m_pad, workspace):
    m, f = g.shape
    gd, ud = _to_dev(g), _to_dev(u)
    hw = torch.full((m, f), 0x5555, dtype=torch.int16, device="cuda") if workspace else None
    q = torch.full((m_pad, f // 2), CANARY, dtype=torch.uint8, device="cuda")
    sfa = torch.full((h3.sf_bytes(m_pad, f),), CANARY, dtype=torch.uint8, device="cuda")
    ts, q, sfa = h3.swiglu_pack(gd, ud, m_pad, h_workspace=hw, qdata=q, sfa=sfa)
    torch.cuda.synchronize()
    assert h3.h3fp4_device_error() == 0
    return float(ts.item()), q.cpu().numpy(), sfa.cpu().numpy(), (None if hw is None else _u16(hw))


def test_silu_exhaustive_over_all_bf16_gates(h3):
    """h = silu_bf16(g) * 1 for every one of the 65,536 bf16 gate patterns."""
    g = np.arange(65536, dtype=np.uint16).reshape(256, 256)
    u = np.full((256, 256), 0x3F80, dtype=np.uint16)         # up = 1.0
    _, _, _, h = run_swiglu(h3, g, u, 256, workspace=True)
    want = oracle.silu_table().reshape(256, 256)
    nan_w = (want & 0x7FFF) > 0x7F80
    nan_h = (h & 0x7FFF) > 0x7F80
    assert np.array_equal(nan_h, nan_w)
    bad = np.argwhere((h != want) & ~nan_w)
    assert bad.size == 0, [(hex(int(g[i, j])), hex(int(h[i, j])), hex(int(want[i, j]))) for i, j in bad[:8]]


@pytest.mark.parametrize("workspace", [False, True])
@pytest.mark.parametrize("m,m_pad,f,scale", [(64, 64, 256, 1.0), (300, 320, 512, 3.0), (129, 256, 768, 20.0)])
def test_swiglu_bit_exact(h3, m, m_pad, f, scale, workspace):
    gen = torch.Generator().manual_seed(m + f)
    g = _bf16(torch.randn(m, f, generator=gen) * scale)
    u = _bf16(torch.randn(m, f, generator=gen))
    ts_o, q_o, sf_o, h_o, _ = oracle.swiglu_producer(g, u, m_pad)
    ts, q, sfa, h = run_swiglu(h3, g, u, m_pad, workspace)
    assert _f32_bits(ts) == _f32_bits(ts_o)
    assert np.array_equal(q, q_o)
    assert np.array_equal(sfa, oracle.swizzle_sf(sf_o))
    if workspace:
        assert np.array_equal(h, h_o)


def run_plain(h3, x, m_pad, ldx=None):
    m, d = x.shape
    ld = d if ldx is None else ldx
    buf = np.zeros((m, ld), dtype=np.uint16)
    buf[:, :d] = x
    xd = _to_dev(buf)[:, :d] if m else torch.empty(0, d, dtype=torch.int16, device="cuda")
    q = torch.full((m_pad, d // 2), CANARY, dtype=torch.uint8, device="cuda")
    sfa = torch.full((h3.sf_bytes(m_pad, d),), CANARY, dtype=torch.uint8, device="cuda")
    ts = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
    h3.quantize_pack(xd, m_pad, tensor_scale=ts, qdata=q, sfa=sfa)
    torch.cuda.synchronize()
    assert h3.h3fp4_device_error() == 0
    return float(ts.item()), q.cpu().numpy(), sfa.cpu().numpy()


def check_plain(h3, x, m_pad, ldx=None):
    ts_o, q_o, sf_o, _ = oracle.plain_producer(x, m_pad)
    ts, q, sfa = run_plain(h3, x, m_pad, ldx)
    assert _f32_bits(ts) == _f32_bits(ts_o), (ts, ts_o)
    assert np.array_equal(q, q_o), f"QDATA differs at {np.argwhere(q != q_o)[:5].tolist()}"
    assert np.array_equal(sfa, oracle.swizzle_sf(sf_o))
    return ts


def test_plain_tiny_adversarial_bit_exact(h3):
    """The adversarial tiny activation (outlier, midpoints, zero and tiny-scale
    blocks, -0 rows, subnormals) packed as it is."""
    from oracle.adversarial import tiny_adversarial
    w = W.WORKLOADS["tiny"]
    a = W.activations(w)
    x = tiny_adversarial(_u16(a["x"]), _u16(a["shift"]), _u16(a["scale"]), W.seg_offsets(w))
    check_plain(h3, x, w.m_pad)


@pytest.mark.parametrize("m,m_pad,d,scale,ldx", [
    (1, 16, 256, 1.0, None), (300, 320, 768, 7.0, None), (129, 256, 512, 0.01, 520), (1000, 1024, 7168, 3.0, None),
])
def test_plain_bit_exact(h3, m, m_pad, d, scale, ldx):
    g = torch.Generator().manual_seed(m + d)
    x = _bf16(torch.randn(m, d, generator=g) * scale)
    x[0, :16] = 0x8000                      # a whole block of -0: scale 0, codes keep the sign
    check_plain(h3, x, m_pad, ldx)


def test_plain_zero_rows(h3):
    ts, q, sfa = run_plain(h3, np.zeros((0, 256), dtype=np.uint16), 16)
    assert ts == 0.0 and not q.any() and not sfa.any()


@pytest.mark.parametrize("m,m_pad,d,off", [
    (0, 16, 256, [0, 0]),
    (1, 16, 256, [0, 1]),
    (300, 320, 768, [0, 0, 150, 300]),
    (16384 + 77, 16512, 4096, [0, 8000, 16461]),      # more tiles than the co-resident grid
])
def test_single_launch_modulation_producer(h3, m, m_pad, d, off):
    """Both passes in one cooperative launch: the same bytes as the oracle (and
    so as the two-call path), every tile packed after the grid barrier."""
    x, sh, sc = _random_case(m, d, len(off) - 1, seed=m + 3 * d)
    ts_o, q_o, sf_o, _, _ = oracle.modulate_producer(x, sh, sc, off, m_pad)
    xd = _to_dev(x) if m else torch.empty(0, d, dtype=torch.int16, device="cuda")
    q = torch.full((m_pad, d // 2), CANARY, dtype=torch.uint8, device="cuda")
    sfa = torch.full((h3.sf_bytes(m_pad, d),), CANARY, dtype=torch.uint8, device="cuda")
    ts = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
    h3.modulate_produce(xd, _to_dev(sh), _to_dev(sc), off, m_pad, tensor_scale=ts, qdata=q, sfa=sfa)
    torch.cuda.synchronize()
    assert h3.h3fp4_device_error() == 0
    assert _f32_bits(float(ts.item())) == _f32_bits(ts_o)
    assert np.array_equal(q.cpu().numpy(), q_o)
    assert np.array_equal(sfa.cpu().numpy(), oracle.swizzle_sf(sf_o))


def test_swizzle_kernel_matches_oracle_layout(h3):
    rng = np.random.default_rng(17)
    for rows, cols in [(384, 16), (300, 64), (1, 4), (129, 896)]:
        sf = rng.integers(0, 256, size=(rows, cols), dtype=np.uint8)
        got = h3.swizzle_scales(torch.from_numpy(sf).cuda()).cpu().numpy()
        pad = np.zeros((h3.sf_rows(rows), cols), dtype=np.uint8)
        pad[:rows] = sf
        assert np.array_equal(got, oracle.swizzle_sf(pad))
