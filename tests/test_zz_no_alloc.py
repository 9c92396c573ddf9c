"""The allocation-free SwiGLU producer, called through the C ABI.

h3fp4_swiglu_pack_noalloc is for callers that cannot allocate device memory
themselves (a plugin inside another framework's operator, a serving loop that
must not allocate after warm-up): it keeps its scratch -- the absmax counters
and the materialised h -- in a static device array owned by the library.  Its
tensor scale, QDATA and scale bytes must equal those of h3fp4_swiglu_pack on
the same inputs, bit for bit (the producer's parity bar), on two calls in a
row with different inputs and sizes, so that the second call shows no trace
of the first one's leftovers in the shared array.  A problem whose h would
not fit the array must be rejected before anything is enqueued.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _inputs(m, f, seed, scale):
    g = torch.Generator().manual_seed(seed)
    gate = (torch.randn(m, f, generator=g) * scale).to(torch.bfloat16).view(torch.int16).cuda()
    up = torch.randn(m, f, generator=g).to(torch.bfloat16).view(torch.int16).cuda()
    return gate, up


def _outputs(h3, m_pad, f):
    ts = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
    q = torch.full((m_pad, f // 2), 0xAB, dtype=torch.uint8, device="cuda")
    sfa = torch.full((h3.sf_bytes(m_pad, f),), 0xAB, dtype=torch.uint8, device="cuda")
    return ts, q, sfa


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _noalloc(h3, gate, up, m_pad):
    m, f = gate.shape
    ts, q, sfa = _outputs(h3, m_pad, f)
    h3.h3fp4_swiglu_pack_noalloc(gate.data_ptr(), f, up.data_ptr(), f, m, m_pad, f, ts.data_ptr(), q.data_ptr(),
                                 sfa.data_ptr(), _stream())
    return ts, q, sfa


def _with_scratch(h3, gate, up, m_pad):
    m, f = gate.shape
    ts, q, sfa = _outputs(h3, m_pad, f)
    scratch = torch.empty(2, dtype=torch.int32, device="cuda")
    h3.h3fp4_swiglu_pack(gate.data_ptr(), f, up.data_ptr(), f, m, m_pad, f, ts.data_ptr(), scratch.data_ptr(),
                         q.data_ptr(), sfa.data_ptr(), None, _stream())
    return ts, q, sfa


def test_noalloc_matches_swiglu_pack_on_two_calls_in_a_row(h3):
    cases = [(1000, 1008, 4096, 1, 2.0),      # 4.1 M elements of h: near the static maximum
             (300, 320, 768, 2, 25.0)]        # smaller, different data: leftovers must not matter
    for m, m_pad, f, seed, scale in cases:
        assert m * f <= h3.NOALLOC_MAX_ELEMENTS
        gate, up = _inputs(m, f, seed, scale)
        a = _noalloc(h3, gate, up, m_pad)
        b = _with_scratch(h3, gate, up, m_pad)
        torch.cuda.synchronize()
        assert h3.h3fp4_device_error() == 0
        ts_a, ts_b = a[0].cpu().numpy(), b[0].cpu().numpy()
        assert ts_a.view(np.uint32)[0] == ts_b.view(np.uint32)[0]
        assert np.array_equal(a[1].cpu().numpy(), b[1].cpu().numpy())
        assert np.array_equal(a[2].cpu().numpy(), b[2].cpu().numpy())


def test_noalloc_rejects_problems_beyond_its_static_scratch(h3):
    f = 1024
    m = h3.NOALLOC_MAX_ELEMENTS // f + 1
    m_pad = -(-m // 16) * 16                   # a valid padding: only the size limit is broken
    gate, up = _inputs(16, f, 3, 1.0)          # real buffers; the size check fails before any use
    ts, q, sfa = _outputs(h3, 16, f)
    with pytest.raises(h3.H3FP4Error) as e:
        h3.h3fp4_swiglu_pack_noalloc(gate.data_ptr(), f, up.data_ptr(), f, m, m_pad, f, ts.data_ptr(),
                                     q.data_ptr(), sfa.data_ptr(), _stream())
    assert e.value.status == 3                 # H3FP4_ERR_SHAPE
    torch.cuda.synchronize()
    assert torch.isnan(ts).all() and (q == 0xAB).all() and (sfa == 0xAB).all()
