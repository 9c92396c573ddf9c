"""Benchmark of the modulation-fused NVFP4 producer + block-scaled GEMM hot path.

One step = the three NVFP4 linears of one DiT block at 37,810 tokens:
  qkv: modulate absmax + modulate pack (K=7168) + GEMM N=21,504
  fc1: modulate absmax + modulate pack (K=7168, MLP shift/scale) + GEMM N=14,336
  fc2: SwiGLU producer (K=14,336) + GEMM N=7,168
The metric is milliseconds per linear (whole job: step time / (3 * ranks)),
lower is better.  Inputs are seeded synthetic tensors resident in HBM; every
input is larger than L2, so no flush is needed between steps.

Also reported: per-kernel CUDA-event times (mean, p50, p95), producer GB/s and
GEMM TFLOP/s with their roofline fractions, an end-to-end number through the
same C-ABI calls with host buffers (host->device copies of the activations and
device->host copies of the outputs inside the timed region), SHA-256 digests
of every linear's inputs and outputs, an AB/BA alternation of two GEMM kernels
on the FC2 linear ("FC2 NVFP4 Library Scheduling", Validation Ladder item 4),
SM clocks sampled during the timed region, and the CPU oracle timed on the
host cores (one core and all cores).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 the script must be launched once per GPU (torch.distributed.run
--nproc-per-node N); every rank runs an independent replica of the step (no
collective on the data path) and the job time is the slowest rank's.
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
from concurrent.futures import ThreadPoolExecutor

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
FP4_PER_BF16 = 13.5 / 2.25        # nominal dense NVFP4 / BF16 tensor rate
NOMINAL_FP4_TFLOPS = 13_500.0     # nominal dense NVFP4 tensor rate
NOMINAL_HBM_GBS = 8_000.0         # nominal HBM3e bandwidth (~8 TB/s)
# Dense E2M1 operations per SM per clock that the FP4 tensor pipe can retire
# (ncu: sm__ops_path_tensor_op_utcomma_src_fp4_dst_fp32_sparsity_off peak_sustained).
FP4_OPS_PER_SM_CLK = 49_152


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
def check_world(gpus: int, world: int) -> None:
    """--gpus must name the number of ranks the launcher started (one per GPU)."""
    if gpus != world:
        raise SystemExit(f"bench.py: --gpus {gpus} but this launch has WORLD_SIZE={world}; run one process per GPU "
                         f"(python -m torch.distributed.run --nproc-per-node {gpus} bench.py --gpus {gpus} ...)")


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


class DeviceTimer:
    """CUDA events on the current stream, synchronised on both sides."""

    def __init__(self):
        import torch
        self.torch = torch
        self.e0 = torch.cuda.Event(enable_timing=True)
        self.e1 = torch.cuda.Event(enable_timing=True)

    def start(self):
        self.torch.cuda.synchronize()
        self.e0.record()

    def stop(self):
        self.e1.record()
        self.torch.cuda.synchronize()

    def elapsed_ms(self):
        return self.e0.elapsed_time(self.e1)


class HostTimer:
    """Wall clock (for CPU stand-ins of the replica path)."""

    def start(self):
        self.t0 = time.perf_counter()

    def stop(self):
        self.t1 = time.perf_counter()

    def elapsed_ms(self):
        return (self.t1 - self.t0) * 1e3


def timed_region(run, timer, world: int, device=None) -> float:
    """Barrier, timer start, run(), timer stop, barrier; the slowest rank's milliseconds."""
    import torch.distributed as dist
    if world > 1:
        dist.barrier()
    timer.start()
    run()
    timer.stop()
    if world > 1:
        dist.barrier()
    return max_over_ranks(timer.elapsed_ms(), device)


# ----------------------------------------------------------------------------
# digests (validation ladder: input and output SHA-256)
# ----------------------------------------------------------------------------
def sha256_of(tensors) -> str:
    h = hashlib.sha256()
    for t in tensors:
        a = t.detach()
        if a.is_cuda:
            a = a.cpu()
        h.update(memoryview(a.contiguous().numpy()).cast("B"))
    return h.hexdigest()


def digests(named):
    """{name: sha256} for a {name: [tensors]} map, hashed in parallel (hashlib releases the GIL)."""
    with ThreadPoolExecutor(max_workers=min(8, max(1, len(named)))) as ex:
        futs = {k: ex.submit(sha256_of, v) for k, v in named.items()}
        return {k: f.result() for k, f in futs.items()}


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
        self.bq, self.bsf_logical = wt["q"], wt["sf"]
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

    def all_inputs(self):
        """Every input of the linear: activations, modulation rows, packed weight, its scales and tensor scale."""
        xs = [self.act[k] for k in sorted(self.act)]
        return xs + [self.bq, self.bsf_logical, self.bts] + ([self.gate, self.res] if self.gated else [])

    def produce(self):
        h3, w, a = self.h3, self.w, self.act
        if w.kind == "modulate":
            h3.modulate_absmax(a["x"], a["shift"], a["scale"], self.off, tensor_scale=self.ts, scratch=self.scratch)
            if self.ev is not None:
                self.ev[3].record()   # between pass 1 and pass 2
            h3.modulate_pack(a["x"], a["shift"], a["scale"], self.off, self.ts, w.m_pad, qdata=self.q, sfa=self.sfa)
        elif w.kind == "plain":
            h3.quantize_pack(a["x"], w.m_pad, tensor_scale=self.ts, scratch=self.scratch, qdata=self.q, sfa=self.sfa)
        else:
            h3.swiglu_pack(a["gate"], a["up"], w.m_pad, h_workspace=self.h, tensor_scale=self.ts,
                           scratch=self.scratch, qdata=self.q, sfa=self.sfa)

    def gemm(self, cfg=None):
        h3, w = self.h3, self.w
        cfg = self.cfg if cfg is None else cfg
        if self.gated:
            h3.gemm_gated_residual(self.q, self.sfa, self.ts, self.bq, self.bsf, self.bts, w.m, self.gate,
                                   self.gate_off, self.res, out=self.c, cfg=cfg)
        else:
            h3.gemm(self.q, self.sfa, self.ts, self.bq, self.bsf, self.bts, w.m, out=self.c, cfg=cfg)

    def run(self, events=None):
        self.ev = events
        if events is not None:
            events[0].record()
        self.produce()
        if events is not None:
            events[1].record()
        self.gemm()
        if events is not None:
            events[2].record()
        self.ev = None


def _pct(xs, q):
    xs = sorted(xs)
    return xs[min(len(xs) - 1, int(round(q * (len(xs) - 1))))]


def ab_ba(h3, L, rounds: int, candidate_kernel: int = 1):
    """Validation ladder item 4 on one linear: baseline (the library's default
    GEMM) and candidate (another GEMM kernel, same arithmetic) alternated AB
    then BA in every round; per arm p50/p95 of the GEMM and of producer+GEMM,
    dense TFLOP/s, workspace bytes and the output SHA-256."""
    import torch
    arms = {"baseline": h3.GemmConfig(0, 0, 0, 0), "candidate": h3.GemmConfig(0, 0, candidate_kernel, 0)}
    times = {a: {"gemm": [], "producer_gemm": []} for a in arms}
    outs = {}

    def one(arm):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record()
        L.produce()
        e[1].record()
        L.gemm(arms[arm])
        e[2].record()
        return e

    for arm in arms:                       # one untimed call of each arm
        one(arm)
    torch.cuda.synchronize()
    recs = []
    for _ in range(rounds):
        for arm in ("baseline", "candidate", "candidate", "baseline"):
            recs.append((arm, one(arm)))
    torch.cuda.synchronize()
    for arm, e in recs:
        times[arm]["gemm"].append(e[1].elapsed_time(e[2]))
        times[arm]["producer_gemm"].append(e[0].elapsed_time(e[2]))
    for arm in arms:
        L.produce()
        L.gemm(arms[arm])
        torch.cuda.synchronize()
        outs[arm] = sha256_of([L.c])
    res = {"linear": L.name, "rounds": rounds, "order": "AB then BA per round",
           "baseline_kernel": GEMM_KERNELS[0], "candidate_kernel": GEMM_KERNELS[candidate_kernel],
           "workspace_bytes": int(L.h.numel() * L.h.element_size()) if L.h is not None else 0}
    for arm in arms:
        g, pg = times[arm]["gemm"], times[arm]["producer_gemm"]
        res[arm] = {"gemm_ms_p50_p95": [round(_pct(g, 0.5), 4), round(_pct(g, 0.95), 4)],
                    "producer_gemm_ms_p50_p95": [round(_pct(pg, 0.5), 4), round(_pct(pg, 0.95), 4)],
                    "gemm_tflops_p50": round(L.flops / (_pct(g, 0.5) * 1e-3) / 1e12, 1),
                    "output_sha256": outs[arm]}
    res["outputs_identical"] = outs["baseline"] == outs["candidate"]
    return res


def run_ours(args, rank, world, local_rank):
    import torch

    import dit_modulate_absmax_gb300 as h3
    from dit_modulate_absmax_gb300 import build as B
    from dit_modulate_absmax_gb300 import workloads as W

    if rank == 0 or not os.path.exists(h3.LIB_PATH):
        B.build()
    if world > 1:
        import torch.distributed as dist
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

    # Each producer alone, back to back (10 runs, median): in the step it follows
    # the previous linear's GEMM, whose ~100 MB of dirty output lines in L2 are
    # written back while pass 1 streams its input; alone, the producer's HBM
    # traffic is its own.
    standalone = {}
    for L in lins:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(11)]
        for e0, e1 in evs:
            e0.record()
            L.produce()
            e1.record()
        torch.cuda.synchronize()
        standalone[L.name] = _pct([e0.elapsed_time(e1) for e0, e1 in evs[1:]], 0.5)
    assert h3.h3fp4_device_error() == 0

    ev = [[[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in lins] for _ in range(args.steps)]

    def timed_steps():
        for k in range(args.steps):
            step(ev[k])

    with ClockSampler(local_rank) as clk:
        if args.profile_range:
            torch.cuda.profiler.start()
        elapsed_ms = timed_region(timed_steps, DeviceTimer(), world, dev)
        if args.profile_range:
            torch.cuda.profiler.stop()
    assert h3.h3fp4_device_error() == 0

    per = {}
    for i, L in enumerate(lins):
        prod = [ev[k][i][0].elapsed_time(ev[k][i][1]) for k in range(args.steps)]
        gem = [ev[k][i][1].elapsed_time(ev[k][i][2]) for k in range(args.steps)]
        per[L.name] = {"producer_ms": sum(prod) / len(prod), "gemm_ms": sum(gem) / len(gem),
                       "producer_p50_p95": (_pct(prod, 0.5), _pct(prod, 0.95)),
                       "gemm_p50_p95": (_pct(gem, 0.5), _pct(gem, 0.95))}
        if L.w.kind == "modulate":   # the two producer passes separately
            p1 = [ev[k][i][0].elapsed_time(ev[k][i][3]) for k in range(args.steps)]
            p2 = [ev[k][i][3].elapsed_time(ev[k][i][1]) for k in range(args.steps)]
            per[L.name]["pass1_ms"] = sum(p1) / len(p1)
            per[L.name]["pass2_ms"] = sum(p2) / len(p2)

    # outputs of the timed steps (device-resident run), kept for the digests
    dev_out = {L.name: ([L.ts.cpu(), L.q.cpu(), L.sfa.cpu()], L.c.cpu()) for L in lins}

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
    # linear.)
    s_in, s_out, s_run = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_run = [torch.cuda.Event() for _ in lins]
    ev_in = [torch.cuda.Event() for _ in lins]
    ev_out = [torch.cuda.Event() for _ in lins]
    started = [False] * len(lins)

    def e2e_step():
        for i, (L, xs_h, out_h) in enumerate(zip(lins, host_in, host_out)):
            with torch.cuda.stream(s_in):
                if started[i]:
                    s_in.wait_event(ev_run[i])
                for xd, xh in zip(L.inputs(), xs_h):
                    xd.copy_(xh, non_blocking=True)
                ev_in[i].record(s_in)
            with torch.cuda.stream(s_run):
                s_run.wait_event(ev_in[i])
                if started[i]:
                    s_run.wait_event(ev_out[i])
                L.run()
                ev_run[i].record(s_run)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_run[i])
                out_h.copy_(L.c, non_blocking=True)
                ev_out[i].record(s_out)
            started[i] = True

    def join_streams():
        cur = torch.cuda.current_stream()
        for s_ in (s_in, s_out, s_run):
            cur.wait_stream(s_)

    def e2e_steps():
        for s_ in (s_in, s_out, s_run):
            s_.wait_stream(torch.cuda.current_stream())
        for _ in range(args.steps):
            e2e_step()
        join_streams()

    for _ in range(max(1, min(args.warmup, 2))):
        e2e_step()
    join_streams()
    e_ms = timed_region(e2e_steps, DeviceTimer(), world, dev)
    assert h3.h3fp4_device_error() == 0

    if rank != 0:
        return None

    # validation-ladder records: digests of every linear's inputs and outputs, and AB/BA on FC2
    named = {}
    for L, out_h in zip(lins, host_out):
        named[f"{L.name}.inputs"] = list(L.all_inputs())
        named[f"{L.name}.producer"] = dev_out[L.name][0]
        named[f"{L.name}.c"] = [dev_out[L.name][1]]
        named[f"{L.name}.e2e"] = [out_h]
    sha = digests(named)
    io_sha = {L.name: {"inputs": sha[f"{L.name}.inputs"],
                       "producer_outputs_ts_qdata_sfa": sha[f"{L.name}.producer"],
                       "gemm_output": sha[f"{L.name}.c"],
                       "e2e_output_identical": sha[f"{L.name}.e2e"] == sha[f"{L.name}.c"]}
              for L in lins}
    ab = None
    if args.ab_rounds > 0:
        target = next((L for L in lins if L.w.kind == "swiglu" and not L.gated), lins[-1])
        ab = ab_ba(h3, target, args.ab_rounds)
        assert h3.h3fp4_device_error() == 0

    peaks = _peaks()
    fp4_peak = peaks["bf16"] * FP4_PER_BF16               # burst: the GEMMs run inside a ~0.1 s region
    fp4_peak_sustained = peaks["bf16_sustained"] * FP4_PER_BF16
    clocks = clk.summary()
    ms_per_step = elapsed_ms / args.steps
    value = job_ms_per_linear(ms_per_step, len(lins), world)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    pipe_peak = (FP4_OPS_PER_SM_CLK * sms * clocks["sm_mhz"] * 1e6 / 1e12) if clocks["sm_mhz"] else None
    kernels = {}
    for L in lins:
        p = per[L.name]
        gbs = L.prod_bytes / (p["producer_ms"] * 1e-3) / 1e9
        tfl = L.flops / (p["gemm_ms"] * 1e-3) / 1e12
        kernels[L.name] = {
            "producer_ms": round(p["producer_ms"], 4), "producer_gbs": round(gbs, 1),
            "producer_hbm_frac": round(gbs / peaks["hbm_gbs"], 4),
            "producer_hbm_frac_nominal": round(gbs / NOMINAL_HBM_GBS, 4),
            "producer_ms_p50_p95": [round(v, 4) for v in p["producer_p50_p95"]],
            "producer_ms_standalone": round(standalone[L.name], 4),
            "producer_hbm_frac_standalone": round(L.prod_bytes / (standalone[L.name] * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
            "gemm_ms": round(p["gemm_ms"], 4), "gemm_tflops": round(tfl, 1),
            "gemm_ms_p50_p95": [round(v, 4) for v in p["gemm_p50_p95"]],
            "epilogue": "gated residual" if L.gated else "bf16",
            "gemm_fp4_frac": round(tfl / fp4_peak, 4),
            "gemm_fp4_frac_nominal": round(tfl / NOMINAL_FP4_TFLOPS, 4)}
        if "pass1_ms" in p:
            kernels[L.name]["pass1_ms"] = round(p["pass1_ms"], 4)
            kernels[L.name]["pass2_ms"] = round(p["pass2_ms"], 4)
    dom = max(lins, key=lambda L: per[L.name]["gemm_ms"])
    dom_ms = per[dom.name]["gemm_ms"]
    achieved = dom.flops / (dom_ms * 1e-3) / 1e12
    out = {
        "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "nvfp4", "data": "synthetic",
        "config": {"workload": WORKLOAD, "m": 37810, "m_pad": 37824, "linears_per_step": len(lins),
                   "l2": "every input larger than L2 (129 MB); no flush", "parallelism": f"replicas{world}"},
        "roofline": {"bound": "tensor",
                     "kernel": f"{GEMM_KERNELS[args.gemm_kernel]} ({dom.name}: M=37810 N={dom.w.n} K={dom.w.k})",
                     "achieved": round(achieved, 1), "peak": round(fp4_peak, 1), "unit": "TFLOP/s",
                     "frac": round(achieved / fp4_peak, 4),
                     "traffic": _profile_traffic(dom.name) if args.gemm_kernel in (0, 4) else None,
                     "peak_source": f"{peaks['source']} bf16 burst {peaks['bf16']} TFLOP/s x {FP4_PER_BF16:g} "
                                    f"(nominal NVFP4/BF16 ratio), of {peaks['source']}",
                     "frac_of_sustained_peak": round(achieved / fp4_peak_sustained, 4),
                     "frac_of_nominal_13500": round(achieved / NOMINAL_FP4_TFLOPS, 4),
                     "frac_of_fp4_pipe_at_run_clock": round(achieved / pipe_peak, 4) if pipe_peak else None},
        "kernels": kernels,
        "hbm_peak_gbs": peaks["hbm_gbs"],
        "e2e": {"value": round(job_ms_per_linear(e_ms / args.steps, len(lins), world), 4), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": sum(L.launches for L in lins) * args.steps,
        "clocks": clocks,
        "sha256": io_sha,
    }
    if ab is not None:
        out["ab_ba"] = ab
    if world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline_both(args.cpu_rows, args.cpu_cols)
    return out


# ----------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)
# ----------------------------------------------------------------------------
def _time_linear_sample(name, rows, cols):
    """Oracle times (s) of each step of one linear on a sample: the producer of
    `rows` rows; the GEMM reference's activation side (dequantising those rows,
    one call per row as gemm_reference does, and |A|); its weight side for
    `cols` weight rows (gemm_reference with no activation rows: dequantising the
    weights and |B|); and its two FP64 products (A B^T and |A| |B|^T) of
    rows x cols outputs."""
    import oracle
    from dit_modulate_absmax_gb300 import workloads as W
    w = W.WORKLOADS[name]
    c = min(cols, w.n)
    act = W.activations(w, device="cpu", m=rows)
    wt = W.weights(w, device="cpu")
    qb, sfb = wt["q"].numpy()[:c], wt["sf"].numpy()[:c]
    t0 = time.perf_counter()
    if w.kind == "modulate":
        ts, q, sf, _, _ = oracle.modulate_producer(act["x"].numpy(), act["shift"].numpy(), act["scale"].numpy(),
                                                   W.seg_offsets(w, rows), rows)
    elif w.kind == "plain":
        ts, q, sf, _ = oracle.plain_producer(act["x"].numpy(), rows)
    else:
        ts, q, sf, _, _ = oracle.swiglu_producer(act["gate"].numpy(), act["up"].numpy(), rows)
    t1 = time.perf_counter()
    A = np.stack([oracle.dequant(q, sf, w.k, ts, r, r + 1)[0] for r in range(rows)])
    Aabs = np.abs(A)
    t2 = time.perf_counter()
    oracle.gemm_reference(q, sf, ts, qb, sfb, wt["ts"], w.k, rows=np.arange(0))
    t3 = time.perf_counter()
    B = oracle.dequant(qb, sfb, w.k, wt["ts"], 0, c)
    Babs = np.abs(B)
    t4 = time.perf_counter()
    _ = A @ B.T
    _ = Aabs @ Babs.T
    t5 = time.perf_counter()
    return {"producer": t1 - t0, "a_side": t2 - t1, "b_side": t3 - t2, "products": t5 - t4, "cols": c}


def _whole_producer_ms(name):
    """The oracle's producer on every row of one linear (the extrapolation check)."""
    import oracle
    from dit_modulate_absmax_gb300 import workloads as W
    w = W.WORKLOADS[name]
    act = W.activations(w, device="cpu")
    t0 = time.perf_counter()
    if w.kind == "modulate":
        oracle.modulate_producer(act["x"].numpy(), act["shift"].numpy(), act["scale"].numpy(), W.seg_offsets(w),
                                 w.m_pad)
    elif w.kind == "plain":
        oracle.plain_producer(act["x"].numpy(), w.m_pad)
    else:
        oracle.swiglu_producer(act["gate"].numpy(), act["up"].numpy(), w.m_pad)
    return (time.perf_counter() - t0) * 1e3


def cpu_sample(rows, cols, whole_producer=False, check_sizes=True):
    """The oracle as it stands on one bounded sample of every linear,
    extrapolated to the full linears step by step: producer and activation side
    x M/rows, weight side x N/cols, FP64 products x (M/rows)(N/cols).  The
    sample runs twice and the faster time of each step is kept (a first call
    pays for thread start-up).  A half-size sample (rows/2, cols/2) reports each step's per-unit rate at the
    smaller size (FP64 matmul is less efficient on smaller matrices, so the
    products' extrapolation from the larger sample errs on the slow side).
    whole_producer: also run the first linear's producer on all of its rows
    and compare with its extrapolation.  check_sizes=False: the full-size
    sample only (the reference arm's steps)."""
    import oracle
    from dit_modulate_absmax_gb300 import workloads as W
    oracle.build()
    oracle.silu_table()
    total_ms, check = 0.0, {}
    for name in LINEARS:
        w = W.WORKLOADS[name]
        sizes = ((rows, cols), (rows // 2, cols // 2)) if check_sizes else ((rows, cols),)
        runs = [[_time_linear_sample(name, r, c) for r, c in sizes] for _ in range(2)]
        full = {k: min(runs[0][0][k], runs[1][0][k]) for k in runs[0][0]}    # twice, the faster one kept
        fm, fn = w.m / rows, w.n / full["cols"]
        total_ms += ((full["producer"] + full["a_side"]) * fm + full["b_side"] * fn + full["products"] * fm * fn) * 1e3
        if not check_sizes:
            continue
        half = {k: min(runs[0][1][k], runs[1][1][k]) for k in runs[0][1]}
        units_full = {"producer": rows, "a_side": rows, "b_side": full["cols"], "products": rows * full["cols"]}
        units_half = {"producer": rows // 2, "a_side": rows // 2, "b_side": half["cols"],
                      "products": (rows // 2) * half["cols"]}
        check[name] = {f"{k}_half_over_full": round((half[k] / units_half[k]) / max(full[k] / units_full[k], 1e-12), 3)
                       for k in units_full}
        if whole_producer and name == LINEARS[0]:
            measured = _whole_producer_ms(name)
            extrapolated = full["producer"] * fm * 1e3
            check["whole_producer"] = {"linear": name, "measured_ms": round(measured, 1),
                                       "extrapolated_ms": round(extrapolated, 1),
                                       "extrapolated_over_measured": round(extrapolated / measured, 3)}
    return total_ms / len(LINEARS), check


def _cpu_worker(rows, cols, threads, repeats, whole_producer, check_sizes):
    """Runs in a child process whose BLAS and OpenMP thread counts were fixed at
    start-up; prints one JSON line per sample."""
    import oracle
    oracle.set_threads(threads)
    for i in range(repeats):
        t0 = time.perf_counter()
        value, check = cpu_sample(rows, cols, whole_producer and i == repeats - 1, check_sizes)
        wall_ms = (time.perf_counter() - t0) * 1e3
        print(json.dumps({"value": value, "check": check, "threads": oracle.threads(), "wall_ms": wall_ms}),
              flush=True)


def _cpu_runs(rows, cols, threads, repeats=1, whole_producer=False, check_sizes=True):
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[k] = str(threads)
    env["CUDA_VISIBLE_DEVICES"] = ""
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-worker", "--cpu-rows", str(rows),
                        "--cpu-cols", str(cols), "--cpu-threads", str(threads), "--cpu-repeats", str(repeats)]
                       + (["--cpu-whole-producer"] if whole_producer else [])
                       + ([] if check_sizes else ["--cpu-no-size-check"]),
                       capture_output=True, text=True, env=env, cwd=ROOT)
    if r.returncode != 0:
        raise RuntimeError(f"CPU oracle worker failed:\n{r.stderr[-2000:]}")
    return [json.loads(l) for l in r.stdout.strip().splitlines() if l.startswith("{")]


def _host_cores():
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


def _sample_text(rows, cols):
    return (f"{rows} activation rows x {cols} weight rows of each of {'/'.join(LINEARS)}, the faster of two passes "
            f"(and a half-size sample for the extrapolation check); each oracle step timed on its own and scaled to "
            f"the full linear: "
            f"producer and activation-side dequantisation by M/rows, weight-side dequantisation by N/cols, the two "
            f"FP64 products by both (extrapolated, not a whole-linear run); C oracle loops (OpenMP over rows) and "
            f"numpy FP64 matmul on the stated threads")


def cpu_baseline_both(rows, cols):
    """The oracle on all host cores (the reported baseline) and on one core."""
    cores = _host_cores()
    allc = _cpu_runs(rows, cols, cores, whole_producer=True)[-1]
    one = _cpu_runs(rows, cols, 1)[-1]
    whole = allc["check"]["whole_producer"]
    return {"value": round(allc["value"], 1), "unit": UNIT, "cores": allc["threads"], "kind": "oracle",
            "sample": _sample_text(rows, cols),
            "one_core": {"value": round(one["value"], 1), "cores": one["threads"]},
            "extrapolation_check": {"all_cores": allc["check"], "one_core": one["check"],
                                    "whole_producer_within_10pct": 0.9 <= whole["extrapolated_over_measured"] <= 1.1}}


def run_reference(args, rank):
    """The reference arm: the oracle as it stands, on the host's cores, on the
    same sample definition as our arm's cpu_baseline; one sample per step."""
    if rank != 0:
        return None
    cores = _host_cores()
    runs = _cpu_runs(args.cpu_rows, args.cpu_cols, cores, args.warmup + args.steps, check_sizes=False)[args.warmup:]
    value = statistics.mean(r["value"] for r in runs)
    spread = (max(r["value"] for r in runs) - min(r["value"] for r in runs)) / value
    step_wall_ms = statistics.mean(r["wall_ms"] for r in runs)
    cb = {"value": round(value, 1), "unit": UNIT, "cores": runs[-1]["threads"], "kind": "oracle",
          "sample": _sample_text(args.cpu_rows, args.cpu_cols) + "; one sample (the faster of two passes) per step",
          "step_spread": round(spread, 3)}
    # ms_per_step is the wall time of one timed step (one sample of every linear), the
    # work actually done; value is that sample extrapolated to full linears.
    return {"impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_wall_ms, 1),
            "ms_per_step_is": "wall time of one sample step; value extrapolates the sample to the full linears",
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "m": 37810, "m_pad": 37824, "linears_per_step": len(LINEARS)},
            "extrapolated": True, "cpu_baseline": cb,
            "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--cpu-rows", type=int, default=256)
    ap.add_argument("--cpu-cols", type=int, default=2048)
    ap.add_argument("--cpu-threads", type=int, default=0, help=argparse.SUPPRESS)
    ap.add_argument("--cpu-worker", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--cpu-repeats", type=int, default=1, help=argparse.SUPPRESS)
    ap.add_argument("--cpu-whole-producer", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--cpu-no-size-check", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ab-rounds", type=int, default=4,
                    help="AB/BA rounds of the default and the single-CTA GEMM on the FC2 linear (0: skip)")
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
    if args.cpu_worker:
        _cpu_worker(args.cpu_rows, args.cpu_cols, args.cpu_threads, args.cpu_repeats, args.cpu_whole_producer,
                    not args.cpu_no_size_check)
        return
    args.warmup = max(args.warmup, 3)
    rank = _env_int("RANK", 0)
    world = _env_int("WORLD_SIZE", 1)
    local_rank = _env_int("LOCAL_RANK", 0)
    if args.impl == "reference":
        out = run_reference(args, rank)
    else:
        check_world(args.gpus, world)
        if world > 1:
            import torch
            import torch.distributed as dist
            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl")
        out = run_ours(args, rank, world, local_rank)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
