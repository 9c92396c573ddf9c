"""Runs one hot-path call on synthetic inputs, for profilers.

  python -m dit_modulate_absmax_gb300.profile_case {modulate,swiglu,plain,gemm} [--m M] [--n N] [--k K] [--reps R]
      [--workspace] [--single-launch] [--cta-pair P] [--n-group G]

`modulate` runs both passes of the modulation producer on an [M, K]
activation, `swiglu` the SwiGLU producer on [M, K] gate/up (with
`--workspace`, the form the benchmark times: pass 1 keeps h), `plain` the
plain-activation producer on an [M, K] bf16 activation, `gemm` the
block-scaled GEMM of a packed [M, K] activation with a packed [N, K] weight.
The R timed repetitions run between cudaProfilerStart and cudaProfilerStop
(so `ncu --profile-from-start off` sees only them) after two warm-up calls,
and the mean CUDA-event time per call is printed.
"""
from __future__ import annotations

import argparse
import dataclasses

import torch

import dit_modulate_absmax_gb300 as h3
from dit_modulate_absmax_gb300 import build as B
from dit_modulate_absmax_gb300 import workloads as W


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("op", choices=("modulate", "swiglu", "plain", "gemm"))
    ap.add_argument("--m", type=int, default=W.M_TOKENS)
    ap.add_argument("--n", type=int, default=21504)
    ap.add_argument("--k", type=int, default=7168)
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--cta-pair", type=int, default=0,
                    help="GEMM kernel (h3fp4_gemm_config.cta_pair): 0 default, 1 single CTA, "
                         "4 CTA pair with copied scales")
    ap.add_argument("--n-group", type=int, default=0, help="GEMM N-group (0 = default)")
    ap.add_argument("--single-launch", action="store_true",
                    help="modulate: both passes in one cooperative launch (h3fp4_modulate_produce)")
    ap.add_argument("--workspace", action="store_true",
                    help="swiglu: keep h in a workspace (pass 1 writes it, pass 2 packs from it)")
    a = ap.parse_args()
    B.build()
    dev = torch.device("cuda")
    m_pad = -(-a.m // 16) * 16
    base = W.WORKLOADS[{"swiglu": "fc2", "plain": "h3_attn"}.get(a.op, "qkv")]
    w = dataclasses.replace(base, m=a.m, m_pad=m_pad, k=a.k, n=a.n,
                            seg_off=(0, min(32768, a.m), a.m) if base.kind == "modulate" else ())
    act = W.activations(w, device=dev)
    off = W.seg_offsets(w)
    ts = torch.empty(1, dtype=torch.float32, device=dev)
    scratch = torch.empty(2, dtype=torch.int32, device=dev)
    q = torch.empty(m_pad, a.k // 2, dtype=torch.uint8, device=dev)
    sfa = torch.empty(h3.sf_bytes(m_pad, a.k), dtype=torch.uint8, device=dev)
    if a.op == "swiglu":
        hw = torch.empty(a.m, a.k, dtype=torch.int16, device=dev) if a.workspace else None

        def call():
            h3.swiglu_pack(act["gate"], act["up"], m_pad, h_workspace=hw, tensor_scale=ts, scratch=scratch, qdata=q,
                           sfa=sfa)
    elif a.op == "plain":
        def call():
            h3.quantize_pack(act["x"], m_pad, tensor_scale=ts, scratch=scratch, qdata=q, sfa=sfa)
    else:
        def produce():
            if a.single_launch:
                h3.modulate_produce(act["x"], act["shift"], act["scale"], off, m_pad, tensor_scale=ts,
                                    scratch=scratch, qdata=q, sfa=sfa)
                return
            h3.modulate_absmax(act["x"], act["shift"], act["scale"], off, tensor_scale=ts, scratch=scratch)
            h3.modulate_pack(act["x"], act["shift"], act["scale"], off, ts, m_pad, qdata=q, sfa=sfa)
        call = produce
        if a.op == "gemm":
            produce()
            wt = W.weights(w, device=dev)
            bsf = h3.swizzle_scales(wt["sf"][: a.n])
            bts = torch.tensor([wt["ts"]], dtype=torch.float32, device=dev)
            c = torch.empty(a.m, a.n, dtype=torch.int16, device=dev)
            cfg = h3.GemmConfig(a.n_group, 0, a.cta_pair, 0)

            def call():
                h3.gemm(q, sfa, ts, wt["q"], bsf, bts, a.m, out=c, cfg=cfg)
    for _ in range(2):
        call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.profiler.start()
    e0.record()
    for _ in range(a.reps):
        call()
    e1.record()
    torch.cuda.synchronize()
    torch.cuda.profiler.stop()
    assert h3.h3fp4_device_error() == 0
    extra = f" cta_pair={a.cta_pair} n_group={a.n_group}" if a.op == "gemm" else ""
    print(f"{a.op} m={a.m} n={a.n} k={a.k}{extra}: {e0.elapsed_time(e1) / a.reps:.4f} ms per call")


if __name__ == "__main__":
    main()
