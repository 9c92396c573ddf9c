"""Seeded sweep of random shapes through the whole modulated linear: the
modulation producer (both launch forms) and the GEMM (every kernel, several
tile schedules, an output leading dimension), each case against the oracle.

Per case the rows, padding, width K, output width N, segment cuts, value
scale, GEMM kernel, N-group and ldc are drawn from one seed; the producer's
tensor scale, QDATA and scale buffer must equal the oracle's byte for byte
and every GEMM output must lie within |C - R| <= ulp_bf16(R) + 1e-5 * S of
the oracle's FP64 sums over the oracle's own packed rows.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu
CANARY = 0xAB
CANARY16 = 0x7E7E
KERNELS = (0, 1, 4)


def _bf16(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(
        np.uint16)


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def _case(seed):
    rng = np.random.default_rng(7000 + seed)
    m = int(rng.integers(1, 900))
    m_pad = -(-m // 16) * 16 + 16 * int(rng.integers(0, 3))
    k = 256 * int(rng.integers(1, 7))
    n = 128 * int(rng.integers(1, 7))
    nseg = int(rng.integers(1, 5))
    cuts = np.sort(rng.integers(0, m + 1, size=nseg - 1))
    off = [0] + [int(c) for c in cuts] + [m]
    scale = float(10.0 ** rng.uniform(-3, 3))
    x = _bf16(rng.standard_normal((m, k)) * scale)
    sh = _bf16(rng.standard_normal((nseg, k)) * 0.2 * scale)
    sc = _bf16(rng.standard_normal((nseg, k)) * 0.2)
    qb = rng.integers(0, 256, size=(n, k // 2), dtype=np.uint8)
    sfb = np.zeros((-(-n // 128) * 128, k // 16), dtype=np.uint8)
    sfb[:n] = rng.integers(0x28, 0x50, size=(n, k // 16))
    cfg = dict(cta_pair=int(rng.choice(KERNELS)), n_group=int(rng.integers(0, 4)))
    ldc = n + 8 * int(rng.integers(0, 3))
    single_launch = bool(seed % 2)
    return m, m_pad, k, n, off, x, sh, sc, qb, sfb, cfg, ldc, single_launch


@pytest.mark.parametrize("seed", range(16))
def test_random_shapes_end_to_end(h3, seed):
    m, m_pad, k, n, off, x, sh, sc, qb, sfb, cfg, ldc, single_launch = _case(seed)
    xd, shd, scd = _dev(x), _dev(sh), _dev(sc)
    q = torch.full((m_pad, k // 2), CANARY, dtype=torch.uint8, device="cuda")
    sfa = torch.full((h3.sf_bytes(m_pad, k),), CANARY, dtype=torch.uint8, device="cuda")
    ts = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
    if single_launch:
        h3.modulate_produce(xd, shd, scd, off, m_pad, tensor_scale=ts, qdata=q, sfa=sfa)
    else:
        h3.modulate_absmax(xd, shd, scd, off, tensor_scale=ts)
        h3.modulate_pack(xd, shd, scd, off, ts, m_pad, qdata=q, sfa=sfa)
    ts_b = torch.tensor([2.0 ** -10], dtype=torch.float32, device="cuda")
    cbuf = torch.full((m + 2, ldc), CANARY16, dtype=torch.int16, device="cuda")
    h3.gemm(q, sfa, ts, torch.from_numpy(qb).cuda(), torch.from_numpy(oracle.swizzle_sf(sfb)).cuda(), ts_b, m,
            out=cbuf[:m].as_strided((m, n), (ldc, 1)), cfg=h3.GemmConfig(cfg["n_group"], 0, cfg["cta_pair"], 0))
    torch.cuda.synchronize()
    assert h3.h3fp4_device_error() == 0

    ts_o, q_o, sf_o, _, _ = oracle.modulate_producer(x, sh, sc, off, m_pad)
    assert np.float32(ts.item()).view(np.uint32) == np.float32(ts_o).view(np.uint32), (ts.item(), ts_o)
    assert np.array_equal(q.cpu().numpy(), q_o), "QDATA differs"
    assert np.array_equal(sfa.cpu().numpy(), oracle.swizzle_sf(sf_o)), "scale buffer differs"

    c = cbuf.cpu().numpy().view(np.uint16)
    assert (c[m:] == CANARY16).all() and (c[:m, n:] == CANARY16).all(), "GEMM wrote outside [m, n]"
    R, S = oracle.gemm_reference(q_o, sf_o, ts_o, qb, sfb, 2.0 ** -10, k, rows=np.arange(m))
    ok, err, tol = oracle.gemm_check(c[:m, :n], R, S)
    assert ok.all(), f"{int((~ok).sum())} outputs outside tolerance ({cfg}, m={m} n={n} k={k})"
