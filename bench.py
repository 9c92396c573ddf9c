"""Benchmark of the modulation-fused NVFP4 producer + block-scaled GEMM hot path.

One step = the three NVFP4 linears of one DiT block at 37,810 tokens:
  qkv: modulate absmax + modulate pack (K=7168) + GEMM N=21,504
  fc1: modulate absmax + modulate pack (K=7168, MLP shift/scale) + GEMM N=14,336
  fc2: SwiGLU producer (K=14,336) + GEMM N=7,168
The metric is milliseconds per linear (whole job: step time / (3 * ranks)),
lower is better.  Inputs are seeded synthetic tensors resident in HBM; every
input is larger than L2, so no flush is needed between steps.

Also reported: per-kernel CUDA-event times, producer GB/s and GEMM TFLOP/s
with their roofline fractions, an end-to-end number through the same C-ABI
calls with host buffers (host->device copies of the activations and
device->host copies of the outputs inside the timed region), SM clocks sampled
during the timed region, and the CPU oracle timed on the host cores.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "producer GB/s & NVFP4 GEMM TFLOP/s vs roofline at M=37,810 rows (ms/linear)"
UNIT = "ms/linear"
# Linear sets: the default (the benchmark's configs) and the model's own projection widths.
WIDTHS = {
    "baseline": (("qkv", "fc1", "fc2"),
                 "DiT block NVFP4 linears at M=37,810 (padded 37,824): qkv K=7168 N=21504, "
                 "fc1 K=7168 N=14336 (fused modulate producer), fc2 K=14336 N=7168 (SwiGLU producer)"),
    "h3": (("h3_qkv", "h3_attn", "h3_fc1", "h3_fc2"),
           "DiT block NVFP4 linears at the model's own widths, M=37,810 (padded 37,824): qkv K=5376 N=21504, "
           "attention output K=7168 N=5376 (plain producer), fc1 K=5376 N=14336 (fused modulate producer), "
           "fc2 K=14336 N=5376 (SwiGLU producer)"),
}
LINEARS, WORKLOAD = WIDTHS["baseline"]
FP4_PER_BF16 = 13.5 / 2.25   # nominal dense NVFP4 / BF16 tensor rate


def _env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16": float(p["bf16_tflops"]),
                "bf16_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.gpu_index = str(device_index)
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            self.gpu_index = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        except Exception:
            pass
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_index, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for l in getattr(self, "lines", []):
            p = [v.strip() for v in l.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx.append(float(p[2]))
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------
# profile summary -> traffic of the dominant kernel (only while its source is unchanged)
# ----------------------------------------------------------------------------
# kernel behind each h3fp4_gemm_config.cta_pair value (0 = the library default)
GEMM_KERNELS = {0: "nvf4_gemm_pair_cp_kernel", 1: "nvf4_gemm_kernel<single CTA>", 4: "nvf4_gemm_pair_cp_kernel"}


def _gemm_source_sha():
    h = hashlib.sha256()
    for f in ("gemm.cu", "ptx.cuh"):
        with open(os.path.join(ROOT, "dit_modulate_absmax_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _profile_traffic(linear):
    path = os.path.join(ROOT, "profiles", "gemm_nvf4_traffic.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(r"source_sha256_16:\s*([0-9a-f]+)", text)
    if not m or m.group(1) != _gemm_source_sha():
        return None
    t = re.search(rf"traffic_bytes_per_launch\[{linear}\]:\s*([0-9.eE+]+)", text)
    return float(t.group(1)) if t else None


# ----------------------------------------------------------------------------
# ranks: N replicas, one per GPU, no collective on the data path
# ----------------------------------------------------------------------------
def max_over_ranks(value_ms: float, device=None) -> float:
    """Largest value over all ranks (the job's time is its slowest replica's)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value_ms)
    t = torch.tensor([float(value_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_ms_per_linear(step_ms: float, linears_per_step: int, world: int) -> float:
    """Whole-job milliseconds per linear: every rank runs its own block, so the
    job finishes linears_per_step * world linears per (slowest) step."""
    return step_ms / (linears_per_step * world)


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------
def _bytes_per_element(kind):
    # producer algorithmic bytes per activation element: both passes read the bf16
    # input (SwiGLU: pass 1 reads gate and up and writes h, pass 2 reads h), pass 2
    # writes 0.5 B of QDATA and 1/16 B of scale
    return (4 + 2 + 2 + 0.5 + 1 / 16) if kind == "swiglu" else (2 + 2 + 0.5 + 1 / 16)


GATED = ("h3_attn", "h3_fc2")   # projections whose output enters the residual stream through a gate


class Linear:
    def __init__(self, h3, W, name, dev, gemm_kernel=0, gated=False):
        import torch
        self.h3, self.name = h3, name
        self.w = w = W.WORKLOADS[name]
        self.act = W.activations(w, device=dev)
        self.off = W.seg_offsets(w) if w.kind == "modulate" else None
        wt = W.weights(w, device=dev)
        self.bq = wt["q"]
        self.bsf = h3.swizzle_scales(wt["sf"][: w.n])
        self.bts = torch.tensor([wt["ts"]], dtype=torch.float32, device=dev)
        self.ts = torch.empty(1, dtype=torch.float32, device=dev)
        self.scratch = torch.empty(2, dtype=torch.int32, device=dev)
        self.q = torch.empty(w.m_pad, w.k // 2, dtype=torch.uint8, device=dev)
        self.sfa = torch.empty(h3.sf_bytes(w.m_pad, w.k), dtype=torch.uint8, device=dev)
        self.c = torch.empty(w.m, w.n, dtype=torch.int16, device=dev)
        # SwiGLU: pass 1 materialises h so that pass 2 reads it instead of recomputing silu
        # (the same HBM bytes either way: h written + read = gate and up read once more)
        self.h = torch.empty(w.m, w.k, dtype=torch.int16, device=dev) if w.kind == "swiglu" else None
        self.flops = 2.0 * w.m * w.n * w.k
        self.prod_bytes = _bytes_per_element(w.kind) * w.m * w.k
        # our kernels per run: modulation = absmax kernel + pack kernel + GEMM; the SwiGLU and
        # plain producers run both passes in one cooperative launch (+ GEMM)
        self.launches = 3 if w.kind == "modulate" else 2
        self.cfg = h3.GemmConfig(0, 0, gemm_kernel, 0) if gemm_kernel else None
        # gated residual epilogue: out = RN(res + RN(gate_s * C)), gate per stream segment
        self.gated = gated and name in GATED
        if self.gated:
            g = torch.Generator(device=dev)
            g.manual_seed(w.seed + 200)
            self.gate_off = [0, 32_768, w.m]
            self.gate = torch.randn(2, w.n, generator=g, device=dev).to(torch.bfloat16).view(torch.int16)
            self.res = (torch.randn(w.m, w.n, generator=g, device=dev) * 4).to(torch.bfloat16).view(torch.int16)
        self.ev = None

    def inputs(self):
        return [self.act[k] for k in (("gate", "up") if self.w.kind == "swiglu" else ("x",))]

    def run(self, events=None):
        h3, w, a = self.h3, self.w, self.act
        if events is not None:
            events[0].record()
        if w.kind == "modulate":
            h3.modulate_absmax(a["x"], a["shift"], a["scale"], self.off, tensor_scale=self.ts, scratch=self.scratch)
            if events is not None:
                events[3].record()   # between pass 1 and pass 2
            h3.modulate_pack(a["x"], a["shift"], a["scale"], self.off, self.ts, w.m_pad, qdata=self.q, sfa=self.sfa)
        elif w.kind == "plain":
            h3.quantize_pack(a["x"], w.m_pad, tensor_scale=self.ts, scratch=self.scratch, qdata=self.q, sfa=self.sfa)
        else:
            h3.swiglu_pack(a["gate"], a["up"], w.m_pad, h_workspace=self.h, tensor_scale=self.ts,
                           scratch=self.scratch, qdata=self.q, sfa=self.sfa)
        if events is not None:
            events[1].record()
        if self.gated:
            h3.gemm_gated_residual(self.q, self.sfa, self.ts, self.bq, self.bsf, self.bts, w.m, self.gate,
                                   self.gate_off, self.res, out=self.c, cfg=self.cfg)
        else:
            h3.gemm(self.q, self.sfa, self.ts, self.bq, self.bsf, self.bts, w.m, out=self.c, cfg=self.cfg)
        if events is not None:
            events[2].record()


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import dit_modulate_absmax_gb300 as h3
    from dit_modulate_absmax_gb300 import build as B
    from dit_modulate_absmax_gb300 import workloads as W

    if rank == 0 or not os.path.exists(h3.LIB_PATH):
        B.build()
    if world > 1:
        dist.barrier()
    h3.lib()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    lins = [Linear(h3, W, n, dev, args.gemm_kernel, args.gated) for n in LINEARS]
    torch.cuda.synchronize()

    def step(ev=None):
        for i, L in enumerate(lins):
            L.run(None if ev is None else ev[i])

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert h3.h3fp4_device_error() == 0

    ev = [[[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in lins] for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        if args.profile_range:
            torch.cuda.profiler.start()
        start.record()
        for k in range(args.steps):
            step(ev[k])
        stop.record()
        torch.cuda.synchronize()
        if args.profile_range:
            torch.cuda.profiler.stop()
    if world > 1:
        dist.barrier()
    elapsed_ms = max_over_ranks(start.elapsed_time(stop), dev)
    assert h3.h3fp4_device_error() == 0

    def pct(xs, q):
        xs = sorted(xs)
        return xs[min(len(xs) - 1, int(round(q * (len(xs) - 1))))]

    per = {}
    for i, L in enumerate(lins):
        prod = [ev[k][i][0].elapsed_time(ev[k][i][1]) for k in range(args.steps)]
        gem = [ev[k][i][1].elapsed_time(ev[k][i][2]) for k in range(args.steps)]
        per[L.name] = {"producer_ms": sum(prod) / len(prod), "gemm_ms": sum(gem) / len(gem),
                       "producer_p50_p95": (pct(prod, 0.5), pct(prod, 0.95)),
                       "gemm_p50_p95": (pct(gem, 0.5), pct(gem, 0.95))}
        if L.w.kind == "modulate":   # the two producer passes separately
            p1 = [ev[k][i][0].elapsed_time(ev[k][i][3]) for k in range(args.steps)]
            p2 = [ev[k][i][3].elapsed_time(ev[k][i][1]) for k in range(args.steps)]
            per[L.name]["pass1_ms"] = sum(p1) / len(p1)
            per[L.name]["pass2_ms"] = sum(p2) / len(p2)

    # end to end through the same C-ABI calls with host buffers
    host_in = [[x.cpu().pin_memory() for x in L.inputs()] for L in lins]
    host_out = [torch.empty(L.c.shape, dtype=L.c.dtype, pin_memory=True) for L in lins]
    h2d = sum(x.numel() * x.element_size() for xs in host_in for x in xs)
    d2h = sum(x.numel() * x.element_size() for x in host_out)

    # Uploads, kernels and downloads on separate streams, as a serving loop
    # would issue them: linear i+1's inputs upload and linear i-1's output
    # downloads while linear i computes.  Per linear: its uploads wait until
    # its previous run consumed the inputs, its run waits for the uploads and
    # for the previous downloads of its output.  (Splitting each transfer over
    # two streams per direction measured slower: 7.8 against 6.4 ms per
    # linear; n_split stays 1.)
    n_split = 1
    s_in = [torch.cuda.Stream(dev) for _ in range(n_split)]
    s_out = [torch.cuda.Stream(dev) for _ in range(n_split)]
    s_run = torch.cuda.Stream(dev)
    ev_in = [[torch.cuda.Event() for _ in range(n_split)] for _ in lins]
    ev_run = [torch.cuda.Event() for _ in lins]
    ev_out = [[torch.cuda.Event() for _ in range(n_split)] for _ in lins]
    started = [False] * len(lins)

    def halves(t, j):
        rows = t.shape[0]
        lo, hi = rows * j // n_split, rows * (j + 1) // n_split
        return t[lo:hi]

    def e2e_step():
        for i, (L, xs_h, out_h) in enumerate(zip(lins, host_in, host_out)):
            for j, st in enumerate(s_in):
                with torch.cuda.stream(st):
                    if started[i]:
                        st.wait_event(ev_run[i])
                    for xd, xh in zip(L.inputs(), xs_h):
                        halves(xd, j).copy_(halves(xh, j), non_blocking=True)
                    ev_in[i][j].record(st)
            with torch.cuda.stream(s_run):
                for j in range(n_split):
                    s_run.wait_event(ev_in[i][j])
                    if started[i]:
                        s_run.wait_event(ev_out[i][j])
                L.run()
                ev_run[i].record(s_run)
            for j, st in enumerate(s_out):
                with torch.cuda.stream(st):
                    st.wait_event(ev_run[i])
                    halves(out_h, j).copy_(halves(L.c, j), non_blocking=True)
                    ev_out[i][j].record(st)
            started[i] = True

    def join_streams():
        cur = torch.cuda.current_stream()
        for s_ in s_in + s_out + [s_run]:
            cur.wait_stream(s_)

    for _ in range(max(1, min(args.warmup, 2))):
        e2e_step()
    join_streams()
    torch.cuda.synchronize()
    e_start, e_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    e_start.record()
    for s_ in s_in + s_out + [s_run]:
        s_.wait_stream(torch.cuda.current_stream())
    for _ in range(args.steps):
        e2e_step()
    join_streams()
    e_stop.record()
    torch.cuda.synchronize()
    e_ms = max_over_ranks(e_start.elapsed_time(e_stop), dev)

    if rank != 0:
        return None
    peaks = _peaks()
    fp4_peak = peaks["bf16_sustained"] * FP4_PER_BF16
    ms_per_step = elapsed_ms / args.steps
    value = job_ms_per_linear(ms_per_step, len(lins), world)
    kernels = {}
    for L in lins:
        p = per[L.name]
        gbs = L.prod_bytes / (p["producer_ms"] * 1e-3) / 1e9
        tfl = L.flops / (p["gemm_ms"] * 1e-3) / 1e12
        kernels[L.name] = {
            "producer_ms": round(p["producer_ms"], 4), "producer_gbs": round(gbs, 1),
            "producer_hbm_frac": round(gbs / peaks["hbm_gbs"], 4),
            "producer_ms_p50_p95": [round(v, 4) for v in p["producer_p50_p95"]],
            "gemm_ms": round(p["gemm_ms"], 4), "gemm_tflops": round(tfl, 1),
            "gemm_ms_p50_p95": [round(v, 4) for v in p["gemm_p50_p95"]],
            "epilogue": "gated residual" if L.gated else "bf16",
            "gemm_fp4_frac": round(tfl / fp4_peak, 4)}
        if "pass1_ms" in p:
            kernels[L.name]["pass1_ms"] = round(p["pass1_ms"], 4)
            kernels[L.name]["pass2_ms"] = round(p["pass2_ms"], 4)
    dom = max(lins, key=lambda L: per[L.name]["gemm_ms"])
    dom_ms = per[dom.name]["gemm_ms"]
    achieved = dom.flops / (dom_ms * 1e-3) / 1e12
    clocks = clk.summary()
    out = {
        "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "nvfp4", "data": "synthetic",
        "config": {"workload": WORKLOAD, "m": 37810, "m_pad": 37824, "linears_per_step": len(lins),
                   "l2": "every input larger than L2 (129 MB); no flush", "parallelism": f"replicas{world}"},
        "roofline": {"bound": "tensor",
                     "kernel": f"{GEMM_KERNELS[args.gemm_kernel]} ({dom.name}: M=37810 N={dom.w.n} K={dom.w.k})",
                     "achieved": round(achieved, 1), "peak": round(fp4_peak, 1), "unit": "TFLOP/s",
                     "frac": round(achieved / fp4_peak, 4), "traffic": _profile_traffic(dom.name) if args.gemm_kernel in (0, 4) else None,
                     "peak_source": f"{peaks['source']} bf16 sustained {peaks['bf16_sustained']} TFLOP/s x "
                                    f"{FP4_PER_BF16:g} (nominal NVFP4/BF16 ratio)"},
        "kernels": kernels,
        "hbm_peak_gbs": peaks["hbm_gbs"],
        "e2e": {"value": round(job_ms_per_linear(e_ms / args.steps, len(lins), world), 4), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": sum(L.launches for L in lins) * args.steps,
        "clocks": clocks,
    }
    if world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args.cpu_rows, args.cpu_cols)
    return out


# ----------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)
# ----------------------------------------------------------------------------
def cpu_baseline(rows=64, cols=2048, seed_device="cpu"):
    """The oracle as it stands on a bounded sample of every linear.

    Sample: `rows` activation rows and `cols` weight rows (output columns).
    Timed per linear: the producer (modulation or SwiGLU, absmax, tensor scale,
    pack) of the sample rows; the oracle's GEMM with no activation rows (its
    per-output-column work: weight dequantisation and |B|); and the oracle's
    GEMM of the sample rows.  Extrapolation to the full linear: producer x
    M/rows, per-column work x N/cols, the remaining GEMM time x (M/rows)(N/cols).
    """
    import oracle
    from dit_modulate_absmax_gb300 import workloads as W
    oracle.build()
    oracle.silu_table()
    total_ms = 0.0
    for name in LINEARS:
        w = W.WORKLOADS[name]
        c = min(cols, w.n)
        act = W.activations(w, device=seed_device, m=rows)
        wt = W.weights(w, device=seed_device)
        qb, sfb = wt["q"].numpy()[:c], wt["sf"].numpy()[:c]
        t0 = time.perf_counter()
        if w.kind == "modulate":
            ts, q, sf, _, _ = oracle.modulate_producer(act["x"].numpy(), act["shift"].numpy(),
                                                       act["scale"].numpy(), W.seg_offsets(w, rows), rows)
        elif w.kind == "plain":
            ts, q, sf, _ = oracle.plain_producer(act["x"].numpy(), rows)
        else:
            ts, q, sf, _, _ = oracle.swiglu_producer(act["gate"].numpy(), act["up"].numpy(), rows)
        t1 = time.perf_counter()
        oracle.gemm_reference(q, sf, ts, qb, sfb, wt["ts"], w.k, rows=np.arange(0))   # per-column work only
        t2 = time.perf_counter()
        oracle.gemm_reference(q, sf, ts, qb, sfb, wt["ts"], w.k, rows=np.arange(rows))
        t3 = time.perf_counter()
        fixed = t2 - t1
        mm = max(t3 - t2 - fixed, 0.0)
        total_ms += ((t1 - t0) * w.m / rows + fixed * w.n / c + mm * (w.m / rows) * (w.n / c)) * 1e3
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": round(total_ms / len(LINEARS), 1), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{rows} activation rows x {cols} weight rows of each of {'/'.join(LINEARS)}; producer time "
                      f"scaled by M/rows, per-column GEMM work by N/cols, FP64 products by both; C loops on "
                      f"one core, FP64 matmul through numpy BLAS threads"}


def run_reference(args, rank):
    if rank != 0:
        return None
    samples = []
    for _ in range(args.warmup):
        cpu_baseline(32, 1024)
    for _ in range(args.steps):
        samples.append(cpu_baseline(32, 1024))
    value = sum(s["value"] for s in samples) / len(samples)
    cb = dict(samples[-1])
    cb["value"] = round(value, 1)
    return {"impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(value * len(LINEARS), 1),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "m": 37810, "m_pad": 37824, "linears_per_step": len(LINEARS)},
            "cpu_baseline": cb,
            "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--cpu-rows", type=int, default=128)
    ap.add_argument("--cpu-cols", type=int, default=4096)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--widths", choices=sorted(WIDTHS), default="baseline",
                    help="linear set: the benchmark's configs (default) or the model's own projection widths")
    ap.add_argument("--gated", action="store_true",
                    help="--widths h3: attention output and FC2 use the gated residual epilogue")
    ap.add_argument("--gemm-kernel", type=int, default=0, choices=(0, 1, 4),
                    help="GEMM kernel (h3fp4_gemm_config.cta_pair): 0 library default (4), 1 single CTA, "
                         "4 CTA pair with the scales copied into TMEM by copy warps")
    ap.add_argument("--profile-range", action="store_true",
                    help="bracket the timed steps with cudaProfilerStart/Stop (for ncu --profile-from-start off)")
    args = ap.parse_args()
    global LINEARS, WORKLOAD
    LINEARS, WORKLOAD = WIDTHS[args.widths]
    args.warmup = max(args.warmup, 3)
    rank = _env_int("RANK", 0)
    world = _env_int("WORLD_SIZE", 1)
    local_rank = _env_int("LOCAL_RANK", 0)
    if args.impl == "reference":
        out = run_reference(args, rank)
    else:
        if world > 1:
            import torch
            import torch.distributed as dist
            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        out = run_ours(args, rank, world, local_rank)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
