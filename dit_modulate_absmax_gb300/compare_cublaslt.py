"""The library's default GEMM against cuBLASLt's block-scaled NVFP4 GEMM on
identical operands (a measurement tool; nothing on the library's call path
uses cuBLASLt).

For each chosen linear of the benchmark (M = 37,810): the library's producer
packs the seeded workload's activations; those bytes and the weight operands
go to a scratch directory; then, alternating, h3fp4_gemm (CUDA events, in this
process) and cuBLASLt (``cublaslt_ref``, a separate process reading the same
bytes) are timed in two regimes -- a burst of ``--burst`` calls (~30 ms, the
bench's regime) and a sustained run of ``--sustained`` calls (~0.5 s, long
enough for the power cap to act) -- with nvidia-smi sampling the SM clock,
power and the power-cap flag during each.  The two outputs are compared at
the end: fraction of bit-identical bf16 values and the largest distance in
bf16 steps (two correct FP32 accumulation orders differ by a few steps at
most).

Operands matter for power: the same cuBLASLt call on low-entropy operands
(all codes non-negative) draws less power and holds a higher clock under the
cap than on these random operands, so only same-operand timings are compared.

  python -m dit_modulate_absmax_gb300.compare_cublaslt [--linears qkv,fc1,fc2] [--rounds 2]
"""
from __future__ import annotations

import argparse
import datetime
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

import dit_modulate_absmax_gb300 as h3
from dit_modulate_absmax_gb300 import build as B
from dit_modulate_absmax_gb300 import workloads as W

_HERE = os.path.dirname(os.path.abspath(__file__))


def build_ref() -> str:
    src = os.path.join(_HERE, "cublaslt_ref.cu")
    exe = os.path.join(B.BUILD, "cublaslt_ref")
    if not os.path.exists(exe) or os.path.getmtime(exe) < os.path.getmtime(src):
        os.makedirs(B.BUILD, exist_ok=True)
        subprocess.check_call([B.NVCC, "-O2", "-std=c++17", "-o", exe, src, "-lcublasLt"])
    return exe


class Clocks:
    """nvidia-smi samples (wall time, SM MHz, power W, power-cap flag) every 20 ms."""

    def __enter__(self):
        self.proc = subprocess.Popen(
            ["nvidia-smi", "--query-gpu=timestamp,clocks.sm,power.draw,clocks_event_reasons.sw_power_cap",
             "--format=csv,noheader,nounits", "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
            text=True)
        return self

    def __exit__(self, *a):
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        self.rows = []
        for line in out.splitlines():
            p = [v.strip() for v in line.split(",")]
            try:
                t = datetime.datetime.strptime(p[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                self.rows.append((t, float(p[1]), float(p[2]), p[3].lower() == "active"))
            except (ValueError, IndexError):
                continue

    def window(self, t0, t1):
        s = [r for r in self.rows if t0 <= r[0] <= t1]
        if not s:
            return {"samples": 0}
        return {"samples": len(s), "sm_mhz": statistics.median(r[1] for r in s),
                "power_w": statistics.median(r[2] for r in s), "power_capped": sum(r[3] for r in s) / len(s)}


def prepare(name, dev, tmp):
    w = W.WORKLOADS[name]
    act = W.activations(w, device=dev)
    if w.kind == "modulate":
        off = W.seg_offsets(w)
        ts = h3.modulate_absmax(act["x"], act["shift"], act["scale"], off)
        q, sfa = h3.modulate_pack(act["x"], act["shift"], act["scale"], off, ts, w.m_pad)
    elif w.kind == "plain":
        ts, q, sfa = h3.quantize_pack(act["x"], w.m_pad)
    else:
        ts, q, sfa = h3.swiglu_pack(act["gate"], act["up"], w.m_pad)
    wt = W.weights(w, device=dev)
    bsf = h3.swizzle_scales(wt["sf"][: w.n])
    bts = torch.tensor([wt["ts"]], dtype=torch.float32, device=dev)
    torch.cuda.synchronize()
    m128 = h3.sf_rows(w.m)
    aq = np.zeros((m128, w.k // 2), dtype=np.uint8)
    aq[: w.m_pad] = q.cpu().numpy()
    for fname, arr in (("aq.bin", aq), ("asf.bin", sfa.cpu().numpy()), ("bq.bin", wt["q"].cpu().numpy()),
                       ("bsf.bin", bsf.cpu().numpy())):
        arr.tofile(os.path.join(tmp, fname))
    alpha = float(np.float32(ts.item()) * np.float32(wt["ts"]))
    return w, (q, sfa, ts, wt["q"], bsf, bts), alpha


def time_ours(w, ops, reps):
    q, sfa, ts, bq, bsf, bts = ops
    c = torch.empty(w.m, w.n, dtype=torch.int16, device=q.device)
    for _ in range(2):
        h3.gemm(q, sfa, ts, bq, bsf, bts, w.m, out=c)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    e0.record()
    for _ in range(reps):
        h3.gemm(q, sfa, ts, bq, bsf, bts, w.m, out=c)
    e1.record()
    torch.cuda.synchronize()
    t1 = time.time()
    assert h3.h3fp4_device_error() == 0
    return t0, t1, e0.elapsed_time(e1) / reps, c


def time_ref(exe, tmp, w, alpha, reps, out=None):
    cmd = [exe, tmp, str(w.m), str(w.n), str(w.k), str(reps), repr(alpha)] + ([out] if out else [])
    r = subprocess.run(cmd, capture_output=True, text=True, check=True)
    line = next(l for l in r.stdout.splitlines() if l.startswith("TIMED"))
    _, t0, t1, ms = line.split()
    return float(t0), float(t1), float(ms)


def bf16_step_distance(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """Distance in bf16 steps between two arrays of bf16 patterns (ordered integers)."""
    def ordered(x):
        x = x.astype(np.int64)
        return np.where(x & 0x8000, 0x8000 - (x & 0x7FFF), 0x8000 + x)
    return np.abs(ordered(a_bits) - ordered(b_bits))


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--linears", default="qkv,fc1,fc2")
    ap.add_argument("--rounds", type=int, default=2)
    ap.add_argument("--burst", type=int, default=20)
    ap.add_argument("--sustained", type=int, default=300)
    a = ap.parse_args()
    B.build()
    exe = build_ref()
    dev = torch.device("cuda")
    rows = []
    with tempfile.TemporaryDirectory() as tmp, Clocks() as clk:
        for name in a.linears.split(","):
            w, ops, alpha = prepare(name, dev, tmp)
            for r in range(a.rounds):
                for regime, reps in (("burst", a.burst), ("sustained", a.sustained)):
                    t0, t1, ms, c = time_ours(w, ops, reps)
                    rows.append((name, regime, "h3fp4_gemm", ms, t0, t1))
                    out = os.path.join(tmp, "c_ref.bin") if r == 0 and regime == "burst" else None
                    u0, u1, ums = time_ref(exe, tmp, w, alpha, reps, out)
                    rows.append((name, regime, "cuBLASLt", ums, u0, u1))
                    if out:
                        ref = np.fromfile(out, dtype=np.uint16).reshape(w.m, w.n)
                        ours = c.cpu().numpy().view(np.uint16)
                        d = bf16_step_distance(ours, ref)
                        print(f"{name}: outputs identical {float((d == 0).mean()):.4f}, max distance {int(d.max())} "
                              f"bf16 steps, 99.9th percentile {float(np.percentile(d, 99.9)):.0f}", flush=True)
            del ops
            torch.cuda.empty_cache()
    print(f"{'linear':6s} {'regime':9s} {'kernel':11s} {'ms':>8s} {'SM MHz':>7s} {'W':>6s} {'capped':>7s}")
    for name, regime, kern, ms, t0, t1 in rows:
        c = clk.window(t0, t1)
        print(f"{name:6s} {regime:9s} {kern:11s} {ms:8.4f} {c.get('sm_mhz', float('nan')):7.0f} "
              f"{c.get('power_w', float('nan')):6.0f} {c.get('power_capped', float('nan')):7.2f}")


if __name__ == "__main__":
    sys.exit(main())
