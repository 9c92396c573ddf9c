"""Sizes whose byte offsets pass 2^31: 160,000 rows of a 7,168-wide activation
(2.29 GB of bf16; row 149,797 is the first whose offset exceeds 2^31 bytes)
through the modulation producer and the QKV-width GEMM (6.9 GB of output).

The activation is drawn on the device with |x| < 1 and one planted 768, with
zero shift and scale rows (y = x up to the sign of zero), so the tensor scale
is known without reading every row on the host: RN_f32(768 / 2688).  Rows
near the 2^31 boundary, the last rows and random rows are then packed by the
oracle from that scale and compared byte for byte with the GPU's QDATA and
scale buffer, and the GEMM's outputs on the same rows must lie within the
oracle's tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
from dit_modulate_absmax_gb300 import workloads as W

pytestmark = pytest.mark.gpu

M, D, N = 160_000, 7_168, 21_504
PLANT = (M - 5, 7_000)


def _rows():
    first_past = (2 ** 31) // (D * 2) + 1
    rows = [np.arange(first_past - 40, first_past + 40), np.arange(M - 300, M),
            np.random.default_rng(41).integers(0, M, size=24), np.array([PLANT[0]])]
    return np.unique(np.concatenate(rows))


def test_offsets_past_2_31_bytes(h3):
    dev = torch.device("cuda")
    g = torch.Generator(device=dev).manual_seed(40)
    x = (torch.rand(M, D, generator=g, device=dev) * 2 - 1).to(torch.bfloat16)
    x[PLANT] = 768.0
    x = x.view(torch.int16)
    zeros = torch.zeros(1, D, dtype=torch.int16, device=dev)
    off = [0, M]
    ts = h3.modulate_absmax(x, zeros, zeros, off)
    q, sfa = h3.modulate_pack(x, zeros, zeros, off, ts, M)
    w = W.WORKLOADS["qkv"]
    wt = W.weights(w, device=dev)
    bsf = h3.swizzle_scales(wt["sf"][:N])
    bts = torch.tensor([wt["ts"]], dtype=torch.float32, device=dev)
    c = h3.gemm(q, sfa, ts, wt["q"], bsf, bts, M)
    torch.cuda.synchronize()
    assert h3.h3fp4_device_error() == 0

    ts_o = oracle.tensor_scale(oracle.bf16_bits(768.0))
    assert np.float32(ts.item()).view(np.uint32) == np.float32(ts_o).view(np.uint32), (ts.item(), ts_o)

    rows = _rows()
    ridx = torch.from_numpy(rows).to(dev)
    x_rows = x[ridx].cpu().numpy().view(np.uint16)
    z = np.zeros((1, D), dtype=np.uint16)
    y_rows = oracle.modulate(x_rows, z, z, [0, len(rows)])
    pad = -(-len(rows) // 16) * 16
    q_o, sf_o = oracle.pack(y_rows, pad, ts_o)
    assert np.array_equal(q[ridx].cpu().numpy(), q_o[: len(rows)]), "QDATA differs"
    sf_all = oracle.unswizzle_sf(sfa.cpu().numpy(), M, D // 16)
    assert np.array_equal(sf_all[rows], sf_o[: len(rows)]), "block scales differ"

    R, S = oracle.gemm_reference(q_o, sf_o, ts_o, wt["q"].cpu().numpy(), wt["sf"].cpu().numpy(), wt["ts"], D,
                                 rows=np.arange(len(rows)))
    ok, err, tol = oracle.gemm_check(c[ridx].cpu().numpy().view(np.uint16), R, S)
    assert ok.all(), f"{int((~ok).sum())} GEMM outputs outside tolerance"
