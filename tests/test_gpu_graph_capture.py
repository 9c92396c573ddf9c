"""The hot path captured into a CUDA graph: after one eager call per device
(which sets the kernels' attributes), the modulation producer (both passes),
the SwiGLU producer and the GEMM enqueue only stream work -- no host
synchronisation, no allocation -- so a whole linear can be captured once and
replayed.  The replays must give the same bytes as eager calls, on fresh inputs
copied into the captured buffers."""
import numpy as np
import pytest
import torch

from dit_modulate_absmax_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _buffers(h3, w, dev):
    act = W.activations(w, device=dev)
    wt = W.weights(w, device=dev)
    return {
        "act": act, "off": W.seg_offsets(w), "bq": wt["q"], "bsf": h3.swizzle_scales(wt["sf"][: w.n]),
        "bts": torch.tensor([wt["ts"]], dtype=torch.float32, device=dev),
        "ts": torch.empty(1, dtype=torch.float32, device=dev), "scratch": torch.empty(2, dtype=torch.int32, device=dev),
        "q": torch.empty(w.m_pad, w.k // 2, dtype=torch.uint8, device=dev),
        "sfa": torch.empty(h3.sf_bytes(w.m_pad, w.k), dtype=torch.uint8, device=dev),
        "c": torch.empty(w.m, w.n, dtype=torch.int16, device=dev),
    }


def _linear(h3, w, b):
    a = b["act"]
    h3.modulate_absmax(a["x"], a["shift"], a["scale"], b["off"], tensor_scale=b["ts"], scratch=b["scratch"])
    h3.modulate_pack(a["x"], a["shift"], a["scale"], b["off"], b["ts"], w.m_pad, qdata=b["q"], sfa=b["sfa"])
    h3.gemm(b["q"], b["sfa"], b["ts"], b["bq"], b["bsf"], b["bts"], w.m, out=b["c"])


def _snapshot(b):
    return [t.clone() for t in (b["ts"], b["q"], b["sfa"], b["c"])]


def test_modulated_linear_and_swiglu_producer_replay_from_a_graph(h3):
    dev = torch.device("cuda")
    w = W.WORKLOADS["tiny"]
    b = _buffers(h3, w, dev)
    g_in = torch.randn(64, 512, generator=torch.Generator().manual_seed(71)).to(torch.bfloat16).view(torch.int16).to(dev)
    u_in = torch.randn(64, 512, generator=torch.Generator().manual_seed(72)).to(torch.bfloat16).view(torch.int16).to(dev)
    sw = {"ts": torch.empty(1, dtype=torch.float32, device=dev), "scratch": torch.empty(2, dtype=torch.int32, device=dev),
          "q": torch.empty(64, 256, dtype=torch.uint8, device=dev),
          "sfa": torch.empty(h3.sf_bytes(64, 512), dtype=torch.uint8, device=dev)}

    def step():
        _linear(h3, w, b)
        h3.swiglu_pack(g_in, u_in, 64, tensor_scale=sw["ts"], scratch=sw["scratch"], qdata=sw["q"], sfa=sw["sfa"])

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()                                   # eager: sets the kernels' attributes once per device
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step()
    torch.cuda.synchronize()

    for seed in (3, 4):                         # fresh inputs through the captured buffers
        gen = torch.Generator(device=dev)
        gen.manual_seed(seed)
        b["act"]["x"].copy_((torch.randn(w.m, w.k, generator=gen, device=dev) * seed).to(torch.bfloat16).view(torch.int16))
        g_in.copy_(torch.randn(64, 512, generator=gen, device=dev).to(torch.bfloat16).view(torch.int16))
        graph.replay()
        torch.cuda.synchronize()
        got = _snapshot(b) + [sw["ts"].clone(), sw["q"].clone(), sw["sfa"].clone()]
        step()                                   # eager on the same inputs
        torch.cuda.synchronize()
        want = _snapshot(b) + [sw["ts"].clone(), sw["q"].clone(), sw["sfa"].clone()]
        for gt, wt in zip(got, want):
            assert torch.equal(gt, wt)
        assert h3.h3fp4_device_error() == 0
