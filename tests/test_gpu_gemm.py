"""GPU parity of the tcgen05 block-scaled NVFP4 GEMM against the CPU oracle.

Outputs must satisfy |C - R| <= ulp_bf16(R) + 1e-5 * sum_k |a_k b_k| with R the
oracle's FP64 sum of dequantised products; where every product and partial
sum is exactly representable in FP32 and alpha is a power of two, C must equal
RN_bf16(R) bit for bit.  Rows >= m and columns of the leading dimension past n
must keep their canary.
"""
import numpy as np
import pytest
import torch

import oracle
from dit_modulate_absmax_gb300 import workloads as W

pytestmark = pytest.mark.gpu
CANARY16 = 0x7E7E

# Every GEMM kernel: one CTA per 128 x 256 tile (cta_pair=1) and CTA pairs on
# 256 x 256 tiles with the scales copied into TMEM by copy warps (cta_pair=4,
# the default).
KERNELS = {"single": 1, "pair_cp": 4}


@pytest.fixture(params=sorted(KERNELS), ids=sorted(KERNELS))
def cfg(request, h3):
    return h3.GemmConfig(0, 0, KERNELS[request.param], 0)


def _rand_operand(rng, rows, k, code_lo, code_hi, sf_rows=None):
    q = rng.integers(0, 256, size=(rows, k // 2), dtype=np.uint8)
    sr = sf_rows if sf_rows is not None else -(-rows // 128) * 128
    sf = np.zeros((sr, k // 16), dtype=np.uint8)
    sf[:rows] = rng.integers(code_lo, code_hi + 1, size=(rows, k // 16))
    return q, sf


def run_gemm(h3, qa, sfa, ts_a, qb, sfb, ts_b, m, ldc=None, extra_rows=3, cfg=None):
    m_pad, kh = qa.shape
    n = qb.shape[0]
    ldc = n if ldc is None else ldc
    a_q = torch.from_numpy(qa).cuda()
    a_sf = torch.from_numpy(oracle.swizzle_sf(sfa)).cuda()
    b_q = torch.from_numpy(qb).cuda()
    b_sf = torch.from_numpy(oracle.swizzle_sf(sfb)).cuda()
    ta = torch.tensor([ts_a], dtype=torch.float32, device="cuda")
    tb = torch.tensor([ts_b], dtype=torch.float32, device="cuda")
    cbuf = torch.full((m + extra_rows, ldc), CANARY16, dtype=torch.int16, device="cuda")
    h3.gemm(a_q, a_sf, ta, b_q, b_sf, tb, m, out=cbuf[:m].as_strided((m, n), (ldc, 1)), cfg=cfg)
    torch.cuda.synchronize()
    assert h3.h3fp4_device_error() == 0
    c = cbuf.cpu().numpy().view(np.uint16)
    assert (c[m:] == CANARY16).all(), "GEMM wrote rows >= m"
    assert (c[:m, n:] == CANARY16).all(), "GEMM wrote columns >= n"
    return c[:m, :n]


def check_tolerance(C, R, S):
    ok, err, tol = oracle.gemm_check(C, R, S)
    bad = np.argwhere(~ok)
    assert bad.size == 0, (f"{len(bad)} outputs outside tolerance; first {bad[:4].tolist()}, "
                           f"err {err[~ok][:4]}, tol {tol[~ok][:4]}")
    return err / tol


def test_exact_products_are_bit_exact(h3, cfg):
    """Power-of-two scales: every product and partial sum is exact, so C = RN_bf16(R)."""
    rng = np.random.default_rng(20)
    m, m_pad, n, k = 200, 256, 384, 512
    # scales 0.25 .. 1: |a_k b_k| <= 36 in steps of 2^-6, so any partial sum of 512
    # terms stays below 2^15 and is exact in FP32 whatever the summation order
    pow2 = np.array([0x28, 0x30, 0x38], dtype=np.uint8)
    qa = rng.integers(0, 256, size=(m_pad, k // 2), dtype=np.uint8)
    qa[m:] = 0
    qb = rng.integers(0, 256, size=(n, k // 2), dtype=np.uint8)
    sfa = np.zeros((256, k // 16), dtype=np.uint8)
    sfb = np.zeros((384, k // 16), dtype=np.uint8)
    sfa[:m] = rng.choice(pow2, size=(m, k // 16))
    sfb[:n] = rng.choice(pow2, size=(n, k // 16))
    ts_a, ts_b = 0.125, 4.0                                               # alpha = 0.5
    C = run_gemm(h3, qa, sfa, ts_a, qb, sfb, ts_b, m, cfg=cfg)
    R, S = oracle.gemm_reference(qa, sfa, ts_a, qb, sfb, ts_b, k, rows=np.arange(m))
    want = np.vectorize(oracle.bf16_bits)(R).astype(np.uint16)
    bad = np.argwhere(C != want)
    assert bad.size == 0, f"{len(bad)} mismatches, first {bad[:4].tolist()}"


@pytest.mark.parametrize("kernel", sorted(KERNELS))
@pytest.mark.parametrize("n_group", [1, 2, 3, 5])
def test_tile_schedules_are_bit_exact(h3, kernel, n_group):
    """Every N-group size visits every output tile once: groups of n_group N-tiles
    sweep M forwards and backwards in turn (a ragged last group included), with
    5 M-tiles (the last partial) and 5 N-tiles of 256 columns.  Power-of-two
    scales keep every sum exact, so C = RN_bf16(R) bit for bit."""
    rng = np.random.default_rng(30 + n_group)
    m, m_pad, n, k = 1100, 1104, 1280, 512
    pow2 = np.array([0x28, 0x30, 0x38], dtype=np.uint8)
    qa = rng.integers(0, 256, size=(m_pad, k // 2), dtype=np.uint8)
    qa[m:] = 0
    qb = rng.integers(0, 256, size=(n, k // 2), dtype=np.uint8)
    sfa = np.zeros((h3.sf_rows(m_pad), k // 16), dtype=np.uint8)
    sfb = np.zeros((n, k // 16), dtype=np.uint8)
    sfa[:m] = rng.choice(pow2, size=(m, k // 16))
    sfb[:] = rng.choice(pow2, size=(n, k // 16))
    cfg = h3.GemmConfig(n_group, 0, KERNELS[kernel], 0)
    C = run_gemm(h3, qa, sfa, 0.5, qb, sfb, 0.25, m, cfg=cfg)
    R, _ = oracle.gemm_reference(qa, sfa, 0.5, qb, sfb, 0.25, k, rows=np.arange(m))
    want = np.vectorize(oracle.bf16_bits)(R).astype(np.uint16)
    bad = np.argwhere(C != want)
    assert bad.size == 0, f"{len(bad)} mismatches, first {bad[:4].tolist()}"


@pytest.mark.parametrize("m,m_pad,n,k", [
    (1, 16, 128, 256),
    (130, 144, 256, 768),
    (300, 320, 384, 256),
    (513, 528, 640, 1024),
    (128, 128, 512, 2048),
])
def test_random_shapes_within_tolerance(h3, cfg, m, m_pad, n, k):
    rng = np.random.default_rng(m * 7 + n + k)
    qa, sfa = _rand_operand(rng, m_pad, k, 0x28, 0x50)
    qa[m:] = 0
    sfa[m:] = 0
    qb, sfb = _rand_operand(rng, n, k, 0x28, 0x50)
    C = run_gemm(h3, qa, sfa, 0.0123, qb, sfb, 2.0 ** -10, m, cfg=cfg)
    R, S = oracle.gemm_reference(qa, sfa, 0.0123, qb, sfb, 2.0 ** -10, k, rows=np.arange(m))
    check_tolerance(C, R, S)


def test_leading_dimension_of_c(h3, cfg):
    rng = np.random.default_rng(22)
    m, m_pad, n, k, ldc = 100, 112, 256, 512, 264
    qa, sfa = _rand_operand(rng, m_pad, k, 0x30, 0x48)
    qb, sfb = _rand_operand(rng, n, k, 0x30, 0x48)
    C = run_gemm(h3, qa, sfa, 1.0, qb, sfb, 1.0, m, ldc=ldc, cfg=cfg)
    R, S = oracle.gemm_reference(qa, sfa, 1.0, qb, sfb, 1.0, k, rows=np.arange(m))
    check_tolerance(C, R, S)


def test_tiny_workload_end_to_end(h3, cfg):
    """Adversarial tiny producer on the GPU, then the GEMM, against the oracle's whole chain."""
    from oracle.adversarial import tiny_adversarial
    w = W.WORKLOADS["tiny"]
    a = W.activations(w)
    off = W.seg_offsets(w)
    sh = a["shift"].numpy().view(np.uint16)
    sc = a["scale"].numpy().view(np.uint16)
    x = tiny_adversarial(a["x"].numpy().view(np.uint16), sh, sc, off)
    ts_o, q_o, sf_o, _, _ = oracle.modulate_producer(x, sh, sc, off, w.m_pad)
    wt = W.weights(w)

    xd = torch.from_numpy(x.view(np.int16)).cuda()
    ts = h3.modulate_absmax(xd, a["shift"].cuda(), a["scale"].cuda(), off)
    q, sfa = h3.modulate_pack(xd, a["shift"].cuda(), a["scale"].cuda(), off, ts, w.m_pad)
    bq = wt["q"].cuda()
    bsf = h3.swizzle_scales(wt["sf"][: w.n].cuda())
    bts = torch.tensor([wt["ts"]], dtype=torch.float32, device="cuda")
    C = h3.gemm(q, sfa, ts, bq, bsf, bts, w.m, cfg=cfg)
    torch.cuda.synchronize()
    R, S = oracle.gemm_reference(q_o, sf_o, ts_o, wt["q"].numpy(), wt["sf"].numpy(), wt["ts"], w.k,
                                 rows=np.arange(w.m))
    check_tolerance(C.cpu().numpy().view(np.uint16), R, S)


def test_zero_rows_writes_nothing(h3, cfg):
    rng = np.random.default_rng(23)
    qa, sfa = _rand_operand(rng, 16, 256, 0x30, 0x40)
    qb, sfb = _rand_operand(rng, 128, 256, 0x30, 0x40)
    run_gemm(h3, qa, sfa, 1.0, qb, sfb, 1.0, 0, extra_rows=4, cfg=cfg)


def test_scale_atom_rows_are_not_mixed(h3, cfg):
    """Rows i and columns j get only their own scales: one nonzero scale row per operand."""
    rng = np.random.default_rng(24)
    m, m_pad, n, k = 256, 256, 256, 512
    qa = rng.integers(0, 256, size=(m_pad, k // 2), dtype=np.uint8)
    qb = rng.integers(0, 256, size=(n, k // 2), dtype=np.uint8)
    sfa = np.zeros((256, k // 16), dtype=np.uint8)
    sfb = np.zeros((256, k // 16), dtype=np.uint8)
    for r in (0, 37, 95, 130, 255):
        sfa[r] = 0x38
    for c in (1, 64, 127, 128, 200):
        sfb[c, 3] = 0x40            # only scale column 3 (K elements 48..63) of these rows
    C = run_gemm(h3, qa, sfa, 1.0, qb, sfb, 1.0, m, cfg=cfg)
    R, S = oracle.gemm_reference(qa, sfa, 1.0, qb, sfb, 1.0, k, rows=np.arange(m))
    nz = np.argwhere(R != 0)
    assert set(map(int, np.unique(nz[:, 0]))) <= {0, 37, 95, 130, 255}
    check_tolerance(C, R, S)


# ---------------------------------------------------------------------------
# Gated residual epilogue ("NVFP4 Streaming Design", P4)
# ---------------------------------------------------------------------------
GATED_KERNELS = {"single": 1, "pair_cp": 4}


def _gated_inputs(rng, m, n, nseg):
    gate = torch.randn(nseg, n, generator=torch.Generator().manual_seed(int(rng.integers(1 << 30))))
    res = torch.randn(m, n, generator=torch.Generator().manual_seed(int(rng.integers(1 << 30)))) * 4
    return (gate.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16),
            res.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))


def run_gated(h3, qa, sfa, ts_a, qb, sfb, ts_b, m, gate, off, res, cfg, in_place=False, extra_rows=3):
    m_pad, kh = qa.shape
    n = qb.shape[0]
    dev = "cuda"
    a = torch.from_numpy(qa).to(dev)
    asf = h3.swizzle_scales(torch.from_numpy(sfa).to(dev))
    b = torch.from_numpy(qb).to(dev)
    bsf = h3.swizzle_scales(torch.from_numpy(sfb).to(dev))
    ta = torch.tensor([ts_a], dtype=torch.float32, device=dev)
    tb = torch.tensor([ts_b], dtype=torch.float32, device=dev)
    g = torch.from_numpy(gate.view(np.int16)).to(dev)
    buf = torch.full((m + extra_rows, n), CANARY16, dtype=torch.int16, device=dev)
    r = buf[:m]
    r.copy_(torch.from_numpy(res.view(np.int16)))
    if in_place:
        h3.gemm_gated_residual(a, asf, ta, b, bsf, tb, m, g, off, r, out=r, cfg=cfg)
        out = buf
    else:
        out = torch.full((m + extra_rows, n), CANARY16, dtype=torch.int16, device=dev)
        h3.gemm_gated_residual(a, asf, ta, b, bsf, tb, m, g, off, r, out=out[:m], cfg=cfg)
    torch.cuda.synchronize()
    assert h3.h3fp4_device_error() == 0
    o = out.cpu().numpy().view(np.uint16)
    assert (o[m:] == CANARY16).all(), "rows >= m must not be written"
    if not in_place:
        assert np.array_equal(buf[:m].cpu().numpy().view(np.uint16), res), "the residual must not change"
    return o[:m]


@pytest.fixture(params=sorted(GATED_KERNELS), ids=sorted(GATED_KERNELS))
def gcfg(request, h3):
    return h3.GemmConfig(0, 0, GATED_KERNELS[request.param], 0)


def test_gated_exact_products_bit_exact(h3, gcfg):
    """Power-of-two scales make the GEMM result exact (c = RN_bf16(R)), so the
    whole epilogue is determined: out must equal the oracle bit for bit."""
    rng = np.random.default_rng(50)
    m, m_pad, n, k = 300, 320, 384, 512
    pow2 = np.array([0x28, 0x30, 0x38], dtype=np.uint8)
    qa = rng.integers(0, 256, size=(m_pad, k // 2), dtype=np.uint8)
    qa[m:] = 0
    qb = rng.integers(0, 256, size=(n, k // 2), dtype=np.uint8)
    sfa = np.zeros((384, k // 16), dtype=np.uint8)
    sfb = np.zeros((384, k // 16), dtype=np.uint8)
    sfa[:m] = rng.choice(pow2, size=(m, k // 16))
    sfb[:n] = rng.choice(pow2, size=(n, k // 16))
    off = [0, 200, 300]                      # a segment boundary inside the second M tile
    gate, res = _gated_inputs(rng, m, n, 2)
    got = run_gated(h3, qa, sfa, 0.125, qb, sfb, 4.0, m, gate, off, res, gcfg)
    R, _ = oracle.gemm_reference(qa, sfa, 0.125, qb, sfb, 4.0, k, rows=np.arange(m))
    c = np.vectorize(oracle.bf16_bits)(R).astype(np.uint16)
    want = oracle.gated_residual(c, gate, off, res)
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} mismatches, first {bad[:4].tolist()}"


@pytest.mark.parametrize("in_place", [False, True])
@pytest.mark.parametrize("m,m_pad,n,k,off", [
    (130, 144, 256, 768, [0, 130]),
    (513, 528, 640, 1024, [0, 100, 100, 513]),      # an empty segment
])
def test_gated_random_within_tolerance_bounds(h3, gcfg, m, m_pad, n, k, off, in_place):
    rng = np.random.default_rng(m + n + k)
    qa, sfa = _rand_operand(rng, m_pad, k, 0x28, 0x50)
    qa[m:] = 0
    sfa[m:] = 0
    qb, sfb = _rand_operand(rng, n, k, 0x28, 0x50)
    gate, res = _gated_inputs(rng, m, n, len(off) - 1)
    got = oracle.bf16_to_f64(run_gated(h3, qa, sfa, 0.0123, qb, sfb, 2.0 ** -10, m, gate, off, res, gcfg,
                                       in_place=in_place))
    R, S = oracle.gemm_reference(qa, sfa, 0.0123, qb, sfb, 2.0 ** -10, k, rows=np.arange(m))
    lo, hi = oracle.gated_residual_bounds(R, S, gate, off, res)
    bad = np.argwhere((got < lo) | (got > hi))
    assert bad.size == 0, f"{len(bad)} outputs outside the bounds, first {bad[:4].tolist()}"
