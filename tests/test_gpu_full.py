"""Full-size parity at the 37,810-token workloads, in the launch configuration
the benchmark times: the benchmark's three linears and the model's own four
projection widths.

The oracle recomputes the global tensor scale over the whole activation (a
plain pass in C), packs a sample of rows (the first and last rows of tiles,
the last logical rows and random rows) and evaluates those rows of the GEMM
over every output column; the GPU results must match bit for bit (producer)
and within the GEMM tolerance.  The padding rows must be zero.
"""
import numpy as np
import pytest
import torch

import oracle
from dit_modulate_absmax_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _sample_rows(m, seed):
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 127, 128, 255, 32767, 32768, m - 129, m - 128, m - 2, m - 1]
    return np.unique(np.concatenate([fixed, rng.integers(0, m, size=13)]))


def _check_producer_rows(w, rows, y_rows, ts_o, q_gpu, sf_gpu):
    """Pack the sampled rows with the oracle and compare their bytes."""
    q_o, sf_o = oracle.pack(y_rows, len(rows), ts_o)
    nb = w.k // 16
    sf_logical = oracle.unswizzle_sf(sf_gpu, -(-w.m_pad // 128) * 128, nb)
    assert np.array_equal(q_gpu[rows], q_o[: len(rows)])
    assert np.array_equal(sf_logical[rows], sf_o[: len(rows)])
    assert not q_gpu[w.m:].any(), "padding rows of QDATA must be zero"
    assert not sf_logical[w.m:].any(), "scales of rows >= m must be zero"
    return q_o[: len(rows)], sf_o


def _check_gemm_rows(w, rows, q_o, sf_o, ts_o, wt, C):
    """GEMM rows `rows` against the oracle's own packed rows (never the GPU's bytes)."""
    R, S = oracle.gemm_reference(q_o, sf_o, ts_o, wt["q"].cpu().numpy(), wt["sf"].cpu().numpy(), wt["ts"],
                                 w.k, rows=np.arange(len(rows)))
    ok, err, tol = oracle.gemm_check(C[rows], R, S)
    assert ok.all(), f"{int((~ok).sum())} outputs outside tolerance (max err/tol {float((err / tol).max()):.3g})"
    return float((err / tol).max())


@pytest.mark.parametrize("name", ["qkv", "fc1"])
def test_modulate_linear_full_size(h3, name):
    w = W.WORKLOADS[name]
    dev = torch.device("cuda")
    act = W.activations(w, device=dev)
    off = W.seg_offsets(w)
    wt = W.weights(w, device=dev)
    ts = h3.modulate_absmax(act["x"], act["shift"], act["scale"], off)
    q, sfa = h3.modulate_pack(act["x"], act["shift"], act["scale"], off, ts, w.m_pad)
    bsf = h3.swizzle_scales(wt["sf"][: w.n])
    bts = torch.tensor([wt["ts"]], dtype=torch.float32, device=dev)
    C = h3.gemm(q, sfa, ts, wt["q"], bsf, bts, w.m)
    torch.cuda.synchronize()
    assert h3.h3fp4_device_error() == 0

    x = act["x"].cpu().numpy().view(np.uint16)
    sh = act["shift"].cpu().numpy().view(np.uint16)
    sc = act["scale"].cpu().numpy().view(np.uint16)
    y = oracle.modulate(x, sh, sc, off)
    ts_o = oracle.tensor_scale(oracle.absmax(y))
    assert float(ts.item()) == ts_o
    rows = _sample_rows(w.m, seed=31)
    q_o, sf_o = _check_producer_rows(w, rows, y[rows], ts_o, q.cpu().numpy(), sfa.cpu().numpy())
    _check_gemm_rows(w, rows, q_o, sf_o, ts_o, wt, C.cpu().numpy().view(np.uint16))


def test_swiglu_linear_full_size(h3):
    w = W.WORKLOADS["fc2"]
    dev = torch.device("cuda")
    act = W.activations(w, device=dev)
    wt = W.weights(w, device=dev)
    ts, q, sfa = h3.swiglu_pack(act["gate"], act["up"], w.m_pad)
    bsf = h3.swizzle_scales(wt["sf"][: w.n])
    bts = torch.tensor([wt["ts"]], dtype=torch.float32, device=dev)
    C = h3.gemm(q, sfa, ts, wt["q"], bsf, bts, w.m)
    torch.cuda.synchronize()
    assert h3.h3fp4_device_error() == 0

    h = oracle.swiglu(act["gate"].cpu().numpy().view(np.uint16), act["up"].cpu().numpy().view(np.uint16))
    ts_o = oracle.tensor_scale(oracle.absmax(h))
    assert float(ts.item()) == ts_o
    rows = _sample_rows(w.m, seed=32)
    q_o, sf_o = _check_producer_rows(w, rows, h[rows], ts_o, q.cpu().numpy(), sfa.cpu().numpy())
    _check_gemm_rows(w, rows, q_o, sf_o, ts_o, wt, C.cpu().numpy().view(np.uint16))


# ---------------------------------------------------------------------------
# The model's own projection widths (hidden 5,376, attention 7,168, MLP 14,336)
# ---------------------------------------------------------------------------
def _weights_and_gemm(h3, w, q, sfa, ts, dev):
    wt = W.weights(w, device=dev)
    bsf = h3.swizzle_scales(wt["sf"][: w.n])
    bts = torch.tensor([wt["ts"]], dtype=torch.float32, device=dev)
    C = h3.gemm(q, sfa, ts, wt["q"], bsf, bts, w.m)
    torch.cuda.synchronize()
    assert h3.h3fp4_device_error() == 0
    return wt, C


@pytest.mark.parametrize("name", ["h3_qkv", "h3_fc1"])
def test_model_width_modulate_linear(h3, name):
    w = W.WORKLOADS[name]
    dev = torch.device("cuda")
    act = W.activations(w, device=dev)
    off = W.seg_offsets(w)
    ts = h3.modulate_absmax(act["x"], act["shift"], act["scale"], off)
    q, sfa = h3.modulate_pack(act["x"], act["shift"], act["scale"], off, ts, w.m_pad)
    wt, C = _weights_and_gemm(h3, w, q, sfa, ts, dev)
    y = oracle.modulate(act["x"].cpu().numpy().view(np.uint16), act["shift"].cpu().numpy().view(np.uint16),
                        act["scale"].cpu().numpy().view(np.uint16), off)
    ts_o = oracle.tensor_scale(oracle.absmax(y))
    assert float(ts.item()) == ts_o
    rows = _sample_rows(w.m, seed=33)
    q_o, sf_o = _check_producer_rows(w, rows, y[rows], ts_o, q.cpu().numpy(), sfa.cpu().numpy())
    _check_gemm_rows(w, rows, q_o, sf_o, ts_o, wt, C.cpu().numpy().view(np.uint16))


def test_model_width_attention_output_linear(h3):
    w = W.WORKLOADS["h3_attn"]
    dev = torch.device("cuda")
    act = W.activations(w, device=dev)
    ts, q, sfa = h3.quantize_pack(act["x"], w.m_pad)
    wt, C = _weights_and_gemm(h3, w, q, sfa, ts, dev)
    x = act["x"].cpu().numpy().view(np.uint16)
    ts_o = oracle.tensor_scale(oracle.absmax(x))
    assert float(ts.item()) == ts_o
    rows = _sample_rows(w.m, seed=34)
    q_o, sf_o = _check_producer_rows(w, rows, x[rows], ts_o, q.cpu().numpy(), sfa.cpu().numpy())
    _check_gemm_rows(w, rows, q_o, sf_o, ts_o, wt, C.cpu().numpy().view(np.uint16))


def test_model_width_swiglu_linear(h3):
    w = W.WORKLOADS["h3_fc2"]
    dev = torch.device("cuda")
    act = W.activations(w, device=dev)
    hw = torch.empty(w.m, w.k, dtype=torch.int16, device=dev)
    ts, q, sfa = h3.swiglu_pack(act["gate"], act["up"], w.m_pad, h_workspace=hw)
    wt, C = _weights_and_gemm(h3, w, q, sfa, ts, dev)
    h = oracle.swiglu(act["gate"].cpu().numpy().view(np.uint16), act["up"].cpu().numpy().view(np.uint16))
    ts_o = oracle.tensor_scale(oracle.absmax(h))
    assert float(ts.item()) == ts_o
    assert np.array_equal(hw.cpu().numpy().view(np.uint16), h)
    rows = _sample_rows(w.m, seed=35)
    q_o, sf_o = _check_producer_rows(w, rows, h[rows], ts_o, q.cpu().numpy(), sfa.cpu().numpy())
    _check_gemm_rows(w, rows, q_o, sf_o, ts_o, wt, C.cpu().numpy().view(np.uint16))
