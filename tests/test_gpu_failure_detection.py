"""Failure detection on the GPU without a fault: a bounded wait is made to run
out and must end its kernel with an error code, leave the outputs untouched
and leave the device usable ("NVFP4 Streaming Design", P2: the cooperative
producer's grid barrier with a bounded wait; the GEMM pipeline's waits are
bounded the same way).

The waits that run out here are ones that nothing will ever satisfy (an
arrival target above the grid size; operand loads that are never issued),
given a 2 ms limit.  Each test then runs the normal entry point on the same
device and checks its result against the oracle.
"""
import time

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

ERR_WAIT_FULL, ERR_WAIT_ACC, ERR_WAIT_SCALES, ERR_GRID_WAIT = 2, 4, 16, 256
LIMIT_US = 2000


def _stream():
    return torch.cuda.current_stream().cuda_stream


def test_producer_grid_barrier_wait_runs_out_then_device_recovers(h3):
    m, m_pad, d = 300, 320, 512
    g = torch.Generator().manual_seed(61)
    x = (torch.randn(m, d, generator=g) * 3).to(torch.bfloat16).view(torch.int16)
    xd = x.cuda()
    ts = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
    scratch = torch.zeros(2, dtype=torch.int32, device="cuda")
    q = torch.full((m_pad, d // 2), 0xAB, dtype=torch.uint8, device="cuda")
    sfa = torch.full((h3.sf_bytes(m_pad, d),), 0xAB, dtype=torch.uint8, device="cuda")
    assert h3.h3fp4_device_error() == 0
    t0 = time.perf_counter()
    h3.h3fp4_diag_producer_barrier_timeout(xd.data_ptr(), d, m, m_pad, d, ts.data_ptr(), scratch.data_ptr(),
                                           q.data_ptr(), sfa.data_ptr(), LIMIT_US, _stream())
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert elapsed < 1.0, f"the kernel returned only after {elapsed:.3f} s"
    assert h3.h3fp4_device_error() & ERR_GRID_WAIT
    assert torch.isnan(ts).all(), "the tensor scale must not be written when the barrier gave up"
    assert (q == 0xAB).all() and (sfa == 0xAB).all(), "no tile may be packed when the barrier gave up"

    # the device is usable: the normal call is bit-exact against the oracle
    ts2, q2, sfa2 = h3.quantize_pack(xd, m_pad)
    torch.cuda.synchronize()
    assert h3.h3fp4_device_error() == 0
    ts_o, q_o, sf_o, _ = oracle.plain_producer(x.numpy().view(np.uint16), m_pad)
    assert float(ts2.item()) == ts_o
    assert np.array_equal(q2.cpu().numpy(), q_o)
    assert np.array_equal(sfa2.cpu().numpy(), oracle.swizzle_sf(sf_o))


def test_gemm_pipeline_waits_run_out_then_device_recovers(h3):
    m, m_pad, n, k = 300, 320, 384, 512
    rng = np.random.default_rng(67)
    qa = rng.integers(0, 256, size=(m_pad, k // 2), dtype=np.uint8)
    qb = rng.integers(0, 256, size=(n, k // 2), dtype=np.uint8)
    sfa = np.zeros((h3.sf_rows(m_pad), k // 16), dtype=np.uint8)
    sfa[:m] = rng.integers(0x30, 0x48, size=(m, k // 16))
    sfb = np.zeros((h3.sf_rows(n), k // 16), dtype=np.uint8)
    sfb[:n] = rng.integers(0x30, 0x48, size=(n, k // 16))
    a_q, b_q = torch.from_numpy(qa).cuda(), torch.from_numpy(qb).cuda()
    a_sf, b_sf = torch.from_numpy(oracle.swizzle_sf(sfa)).cuda(), torch.from_numpy(oracle.swizzle_sf(sfb)).cuda()
    ta = torch.tensor([0.125], dtype=torch.float32, device="cuda")
    tb = torch.tensor([0.5], dtype=torch.float32, device="cuda")
    c = torch.full((m, n), 0x7E7E, dtype=torch.int16, device="cuda")
    assert h3.h3fp4_device_error() == 0
    t0 = time.perf_counter()
    h3.h3fp4_diag_gemm_wait_timeout(a_q.data_ptr(), a_sf.data_ptr(), ta.data_ptr(), b_q.data_ptr(), b_sf.data_ptr(),
                                    tb.data_ptr(), c.data_ptr(), n, m, m_pad, n, k, LIMIT_US, _stream())
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert elapsed < 1.0, f"the kernel returned only after {elapsed:.3f} s"
    code = h3.h3fp4_device_error()
    assert code & ERR_WAIT_FULL and code & ERR_WAIT_SCALES and code & ERR_WAIT_ACC, hex(code)
    assert (c == 0x7E7E).all(), "no output may be written when the pipeline gave up"

    # the device is usable: the normal call is within the GEMM tolerance of the oracle
    out = h3.gemm(a_q, a_sf, ta, b_q, b_sf, tb, m)
    torch.cuda.synchronize()
    assert h3.h3fp4_device_error() == 0
    R, S = oracle.gemm_reference(qa, sfa, 0.125, qb, sfb, 0.5, k, rows=np.arange(m))
    ok, err, tol = oracle.gemm_check(out.cpu().numpy().view(np.uint16), R, S)
    assert ok.all(), f"{int((~ok).sum())} outputs outside tolerance"
