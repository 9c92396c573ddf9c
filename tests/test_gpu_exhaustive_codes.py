"""Every finite bf16 value under every E4M3 block scale, and as every block
maximum, through the GPU pack.

For a tensor maximum A (planted in the first block), the blocks are built so
that each one's maximum lands on a chosen E4M3 block scale and its other 15
values run through every finite bf16 pattern whose magnitude does not exceed
that maximum.  Over all 126 non-zero scale codes this puts each finite bf16
value through the E2M1 encoding under each block scale product that can hold
it, for three tensor scales.  The plain producer's QDATA and scale bytes must
equal the oracle's byte for byte.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

D = 7_168


def _finite_bf16():
    p = np.arange(65536, dtype=np.uint32)
    exp = (p >> 7) & 0xFF
    return p[exp != 0xFF].astype(np.uint16)


def _tensor(amax):
    ts = np.float32(oracle.tensor_scale(oracle.bf16_bits(amax)))
    den = np.float32(np.float32(6.0) * ts)
    pats = _finite_bf16()
    mags = np.abs(oracle.bf16_to_f64(pats))
    blocks = [np.concatenate([[oracle.bf16_bits(amax)], np.zeros(15, dtype=np.int64)]).astype(np.uint16)]
    e4m3 = oracle.e4m3_table()
    for code in range(1, 127):
        bmax_bits = oracle.bf16_bits(float(e4m3[code]) * float(den))
        bmax = oracle.bf16_value(bmax_bits)
        if not (0 < bmax <= amax):
            continue
        pool = pats[mags <= bmax]
        pad = (-len(pool)) % 15
        pool = np.concatenate([pool, np.zeros(pad, dtype=np.uint16)]).reshape(-1, 15)
        head = np.full((len(pool), 1), bmax_bits, dtype=np.uint16)
        blocks.append(np.concatenate([head, pool], axis=1).reshape(-1))
    flat = np.concatenate(blocks)
    flat = np.concatenate([flat, np.zeros((-len(flat)) % D, dtype=np.uint16)])
    return flat.reshape(-1, D)


@pytest.mark.parametrize("amax", [1.0, 448.0, 7.5])
def test_every_value_under_every_block_scale(h3, amax):
    x = _tensor(amax)
    m = x.shape[0]
    m_pad = -(-m // 16) * 16
    ts_o, q_o, sf_o, _ = oracle.plain_producer(x, m_pad)
    assert len(np.unique(sf_o[:m])) > 120, "the blocks should span the block scale codes"
    xd = torch.from_numpy(x.view(np.int16)).cuda()
    ts, q, sfa = h3.quantize_pack(xd, m_pad)
    torch.cuda.synchronize()
    assert h3.h3fp4_device_error() == 0
    assert np.float32(ts.item()).view(np.uint32) == np.float32(ts_o).view(np.uint32)
    qg = q.cpu().numpy()
    bad = np.flatnonzero((qg != q_o).any(axis=1))
    assert bad.size == 0, f"QDATA differs in {bad.size} rows (first {bad[:5].tolist()})"
    assert np.array_equal(sfa.cpu().numpy(), oracle.swizzle_sf(sf_o)), "scale bytes differ"


@pytest.mark.parametrize("amax", [1.0, 448.0, 7.5])
def test_every_block_maximum(h3, amax):
    """One block per finite bf16 value v with |v| <= A (v first, then v's
    negation and 14 zeros): every possible block maximum meets the E4M3
    rounding of RN_f32(bamax / RN_f32(6 ts)), midpoints included."""
    pats = _finite_bf16()
    vals = pats[np.abs(oracle.bf16_to_f64(pats)) <= amax]
    blocks = np.zeros((len(vals) + 1, 16), dtype=np.uint16)
    blocks[0, 0] = oracle.bf16_bits(amax)
    blocks[1:, 0] = vals
    blocks[1:, 1] = vals ^ 0x8000
    flat = blocks.reshape(-1)
    x = np.concatenate([flat, np.zeros((-len(flat)) % D, dtype=np.uint16)]).reshape(-1, D)
    m = x.shape[0]
    m_pad = -(-m // 16) * 16
    ts_o, q_o, sf_o, _ = oracle.plain_producer(x, m_pad)
    xd = torch.from_numpy(x.view(np.int16)).cuda()
    ts, q, sfa = h3.quantize_pack(xd, m_pad)
    torch.cuda.synchronize()
    assert h3.h3fp4_device_error() == 0
    assert np.float32(ts.item()).view(np.uint32) == np.float32(ts_o).view(np.uint32)
    assert np.array_equal(q.cpu().numpy(), q_o), "QDATA differs"
    assert np.array_equal(sfa.cpu().numpy(), oracle.swizzle_sf(sf_o)), "scale bytes differ"
