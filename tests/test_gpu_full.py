"""Full-size parity at the 37,810-token workloads, in the launch configuration
the benchmark times: the producer-only workload, the benchmark's three linears
and the model's own four projection widths.

Producer: the oracle recomputes every row (modulation or SwiGLU, the global
absolute maximum, the tensor scale, the E4M3 block scales and E2M1 codes of
all 37,810 rows, and the zero padding up to the scale layout's 128-row
multiple); the GPU's tensor scale, QDATA and scale buffer must equal it byte
for byte, every row and every padding byte included ("NVFP4 Modulation
Producer Fusion", Exactness Contract and Result: byte-identical QDATA and E4M3
block scales for complete 37,810-row inputs).

GEMM: whole 256-row output tiles of the default kernel -- the first, the last
(partial: 178 rows) and the two on either side of the segment boundary at row
32,768 -- plus random rows, over every output column, against the oracle's
FP64 sums of its own packed rows (never the GPU's bytes); each output within
1 bf16 ulp + 1e-5 * sum |a_k b_k|.
"""
import numpy as np
import pytest
import torch

import oracle
from dit_modulate_absmax_gb300 import workloads as W

pytestmark = pytest.mark.gpu

PAIR_TILE_M = 256


def _gemm_rows(m, seed):
    """Rows of whole M tiles (first, last, both sides of row 32,768) plus random rows."""
    last = (m - 1) // PAIR_TILE_M
    tiles = sorted({0, last, 32_768 // PAIR_TILE_M - 1, 32_768 // PAIR_TILE_M})
    rows = [np.arange(t * PAIR_TILE_M, min(m, (t + 1) * PAIR_TILE_M)) for t in tiles]
    rows.append(np.random.default_rng(seed).integers(0, m, size=16))
    return np.unique(np.concatenate(rows))


def _u16(t):
    return t.cpu().numpy().view(np.uint16)


def _check_producer_all_rows(w, y, ts, q, sfa):
    """Every byte of the GPU's producer outputs against the oracle's pack of all rows of y."""
    ts_o = oracle.tensor_scale(oracle.absmax(y))
    got_ts = np.float32(ts.item())
    assert got_ts.view(np.uint32) == np.float32(ts_o).view(np.uint32), (float(got_ts), ts_o)
    q_o, sf_o = oracle.pack(y, w.m_pad, ts_o)
    q_g = q.cpu().numpy()
    bad = np.flatnonzero((q_g != q_o).any(axis=1))
    assert bad.size == 0, f"QDATA differs in {bad.size} of {w.m_pad} rows (first {bad[:5].tolist()})"
    sfa_g = sfa.cpu().numpy()
    sf_g = oracle.unswizzle_sf(sfa_g, sf_o.shape[0], sf_o.shape[1])
    bad = np.flatnonzero((sf_g != sf_o).any(axis=1))
    assert bad.size == 0, f"block scales differ in {bad.size} rows (first {bad[:5].tolist()})"
    assert np.array_equal(sfa_g, oracle.swizzle_sf(sf_o)), "scale buffer differs from the oracle's layout"
    assert not q_o[w.m:].any() and not sf_o[w.m:].any()   # the oracle's own padding reading
    return ts_o, q_o, sf_o


def _gemm(h3, w, q, sfa, ts, dev):
    wt = W.weights(w, device=dev)
    bsf = h3.swizzle_scales(wt["sf"][: w.n])
    bts = torch.tensor([wt["ts"]], dtype=torch.float32, device=dev)
    C = h3.gemm(q, sfa, ts, wt["q"], bsf, bts, w.m)
    torch.cuda.synchronize()
    assert h3.h3fp4_device_error() == 0
    return wt, C


def _check_gemm_rows(w, q_o, sf_o, ts_o, wt, C, seed):
    rows = _gemm_rows(w.m, seed)
    R, S = oracle.gemm_reference(q_o, sf_o, ts_o, wt["q"].cpu().numpy(), wt["sf"].cpu().numpy(), wt["ts"], w.k,
                                 rows=rows)
    got = _u16(C[torch.from_numpy(rows).to(C.device)])
    ok, err, tol = oracle.gemm_check(got, R, S)
    assert ok.all(), f"{int((~ok).sum())} outputs outside tolerance (max err/tol {float((err / tol).max()):.3g})"


def _modulate_y(act, off):
    return oracle.modulate(_u16(act["x"]), _u16(act["shift"]), _u16(act["scale"]), off)


def test_producer_workload_full_size_both_launch_forms(h3):
    """The producer-only configuration (37,810 x 7,168, two segments), through
    the two-launch form (h3fp4_modulate_absmax + h3fp4_modulate_pack) and the
    single cooperative launch (h3fp4_modulate_produce)."""
    w = W.WORKLOADS["producer"]
    dev = torch.device("cuda")
    act = W.activations(w, device=dev)
    off = W.seg_offsets(w)
    ts = h3.modulate_absmax(act["x"], act["shift"], act["scale"], off)
    q, sfa = h3.modulate_pack(act["x"], act["shift"], act["scale"], off, ts, w.m_pad)
    ts1, q1, sfa1 = h3.modulate_produce(act["x"], act["shift"], act["scale"], off, w.m_pad)
    torch.cuda.synchronize()
    assert h3.h3fp4_device_error() == 0
    y = _modulate_y(act, off)
    _check_producer_all_rows(w, y, ts, q, sfa)
    _check_producer_all_rows(w, y, ts1, q1, sfa1)


@pytest.mark.parametrize("name", ["qkv", "fc1", "h3_qkv", "h3_fc1"])
def test_modulate_linear_full_size(h3, name):
    w = W.WORKLOADS[name]
    dev = torch.device("cuda")
    act = W.activations(w, device=dev)
    off = W.seg_offsets(w)
    ts = h3.modulate_absmax(act["x"], act["shift"], act["scale"], off)
    q, sfa = h3.modulate_pack(act["x"], act["shift"], act["scale"], off, ts, w.m_pad)
    wt, C = _gemm(h3, w, q, sfa, ts, dev)
    ts_o, q_o, sf_o = _check_producer_all_rows(w, _modulate_y(act, off), ts, q, sfa)
    _check_gemm_rows(w, q_o, sf_o, ts_o, wt, C, seed=31)


@pytest.mark.parametrize("name,workspace", [("fc2", False), ("h3_fc2", True)])
def test_swiglu_linear_full_size(h3, name, workspace):
    w = W.WORKLOADS[name]
    dev = torch.device("cuda")
    act = W.activations(w, device=dev)
    hw = torch.empty(w.m, w.k, dtype=torch.int16, device=dev) if workspace else None
    ts, q, sfa = h3.swiglu_pack(act["gate"], act["up"], w.m_pad, h_workspace=hw)
    wt, C = _gemm(h3, w, q, sfa, ts, dev)
    h = oracle.swiglu(_u16(act["gate"]), _u16(act["up"]))
    if workspace:
        assert np.array_equal(_u16(hw), h), "materialised h differs from the oracle"
    ts_o, q_o, sf_o = _check_producer_all_rows(w, h, ts, q, sfa)
    _check_gemm_rows(w, q_o, sf_o, ts_o, wt, C, seed=32)


def test_model_width_attention_output_linear(h3):
    w = W.WORKLOADS["h3_attn"]
    dev = torch.device("cuda")
    act = W.activations(w, device=dev)
    ts, q, sfa = h3.quantize_pack(act["x"], w.m_pad)
    wt, C = _gemm(h3, w, q, sfa, ts, dev)
    ts_o, q_o, sf_o = _check_producer_all_rows(w, _u16(act["x"]), ts, q, sfa)
    _check_gemm_rows(w, q_o, sf_o, ts_o, wt, C, seed=34)


def test_model_width_fc2_gated_residual_in_place_full_size(h3):
    """The model-width FC2 (37,810 x 5,376 x 14,336) through the gated residual
    epilogue ("NVFP4 Streaming Design", P4), written in place over the residual
    with two gate segments split at row 32,768, in the benchmark's launch form:
    whole 256-row tiles (first, last, both sides of the split) and random rows,
    every column, within the bounds the oracle derives from its FP64 sums."""
    w = W.WORKLOADS["h3_fc2"]
    dev = torch.device("cuda")
    act = W.activations(w, device=dev)
    ts, q, sfa = h3.swiglu_pack(act["gate"], act["up"], w.m_pad)
    wt = W.weights(w, device=dev)
    bsf = h3.swizzle_scales(wt["sf"][: w.n])
    bts = torch.tensor([wt["ts"]], dtype=torch.float32, device=dev)
    g = torch.Generator().manual_seed(36)
    gate = torch.randn(2, w.n, generator=g).to(torch.bfloat16).view(torch.int16)
    res = (torch.randn(w.m, w.n, generator=g) * 4).to(torch.bfloat16).view(torch.int16)
    off = [0, 32_768, w.m]
    out = res.to(dev)
    h3.gemm_gated_residual(q, sfa, ts, wt["q"], bsf, bts, w.m, gate.to(dev), off, out, out=out)
    torch.cuda.synchronize()
    assert h3.h3fp4_device_error() == 0
    ts_o, q_o, sf_o = _check_producer_all_rows(w, oracle.swiglu(_u16(act["gate"]), _u16(act["up"])), ts, q, sfa)
    rows = _gemm_rows(w.m, seed=37)
    R, S = oracle.gemm_reference(q_o, sf_o, ts_o, wt["q"].cpu().numpy(), wt["sf"].cpu().numpy(), wt["ts"], w.k,
                                 rows=rows)
    res_rows = res.numpy().view(np.uint16)[rows]
    split = int((rows < 32_768).sum())
    lo, hi = oracle.gated_residual_bounds(R, S, gate.numpy().view(np.uint16), [0, split, len(rows)], res_rows)
    got = oracle.bf16_to_f64(_u16(out[torch.from_numpy(rows).to(dev)]))
    bad = np.argwhere((got < lo) | (got > hi))
    assert bad.size == 0, f"{len(bad)} outputs outside the bounds, first {bad[:4].tolist()}"
