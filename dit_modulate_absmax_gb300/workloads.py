"""Seeded synthetic inputs shaped like the DiT block workloads.

This module only draws random numbers: it holds none of the producer's or the
GEMM's arithmetic, and both the CUDA path's tests and the CPU oracle take their
inputs from it.  Random floats are drawn with ``torch.randn`` on the requested
device and rounded to bf16 by torch's own conversion; packed weights are drawn
directly as random E2M1 bytes and random E4M3 codes from a fixed code range, so
no encoder is involved.

Workloads (one DiT block at the 37,810-token shape):

* ``tiny``     -- 300 rows (segments 0-255 / 256-299), D=256, N=384; weights
  with E4M3 codes for values 0.5 ... 4 and weight tensor scale 0.01.
* ``producer`` -- 37,810 x 7,168, segments 0-32,767 / 32,768-37,809, rows drawn
  N(0,1) then divided by their RMS; shift/scale N(0, 0.2); padded to 37,824.
* ``qkv``      -- the producer workload plus weights [21,504, 7,168].
* ``fc1``      -- N(0,1) rows with 0.1% of entries replaced by N(0,30),
  MLP shift/scale, weights [14,336, 7,168].
* ``fc2``      -- gate, up N(0,1) [37,810, 14,336], weights [7,168, 14,336].

The model's own projection widths (hidden width 5,376, attention width 7,168,
MLP width 14,336; QKV output 21,504) at the same 37,810 tokens:

* ``h3_qkv``   -- as ``qkv`` with K=5,376.
* ``h3_attn``  -- attention output: plain N(0,1) activations [37,810, 7,168]
  (quantized without a fused transform), weights [5,376, 7,168].
* ``h3_fc1``   -- as ``fc1`` with K=5,376.
* ``h3_fc2``   -- as ``fc2`` with N=5,376.

Weights (all but ``tiny``) use E4M3 codes for values 0.25 ... 8 and a weight
tensor scale of 2^-10.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

M_TOKENS = 37_810
M_PAD = 37_824


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str                 # "modulate", "swiglu" or "plain"
    m: int                    # logical rows
    m_pad: int                # descriptor rows (zero padded)
    k: int                    # producer width D (= GEMM K)
    n: int                    # GEMM output width (0: producer only)
    seg_off: tuple = ()       # row offsets of the modulation segments
    seed: int = 0
    mod_std: float = 0.2      # std of shift / scale
    outlier_frac: float = 0.0
    outlier_std: float = 0.0
    rms_rows: bool = False
    sf_code_lo: int = 0x28    # E4M3 code range of weight block scales
    sf_code_hi: int = 0x50
    w_ts: float = 2.0 ** -10
    extra: dict = field(default_factory=dict, compare=False)


WORKLOADS = {
    "tiny": Workload("tiny", "modulate", 300, 320, 256, 384, (0, 256, 300), seed=0,
                     mod_std=0.1, sf_code_lo=0x30, sf_code_hi=0x48, w_ts=0.01),
    "producer": Workload("producer", "modulate", M_TOKENS, M_PAD, 7168, 0,
                         (0, 32_768, M_TOKENS), seed=1, rms_rows=True),
    "qkv": Workload("qkv", "modulate", M_TOKENS, M_PAD, 7168, 21_504,
                    (0, 32_768, M_TOKENS), seed=2, rms_rows=True),
    "fc1": Workload("fc1", "modulate", M_TOKENS, M_PAD, 7168, 14_336,
                    (0, 32_768, M_TOKENS), seed=3, outlier_frac=0.001, outlier_std=30.0),
    "fc2": Workload("fc2", "swiglu", M_TOKENS, M_PAD, 14_336, 7_168, (), seed=4),
    "h3_qkv": Workload("h3_qkv", "modulate", M_TOKENS, M_PAD, 5376, 21_504,
                       (0, 32_768, M_TOKENS), seed=5, rms_rows=True),
    "h3_attn": Workload("h3_attn", "plain", M_TOKENS, M_PAD, 7168, 5376, (), seed=6),
    "h3_fc1": Workload("h3_fc1", "modulate", M_TOKENS, M_PAD, 5376, 14_336,
                       (0, 32_768, M_TOKENS), seed=7, outlier_frac=0.001, outlier_std=30.0),
    "h3_fc2": Workload("h3_fc2", "swiglu", M_TOKENS, M_PAD, 14_336, 5376, (), seed=8),
}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _bf16(t: torch.Tensor) -> torch.Tensor:
    """float32 -> bf16 (torch's round-to-nearest-even), returned as int16 patterns."""
    return t.to(torch.bfloat16).view(torch.int16)


def activations(w: Workload, device="cpu", m: int | None = None) -> dict:
    """Producer inputs as int16 bf16 patterns: x [m, k], shift/scale [nseg, k]
    for modulate workloads; gate/up [m, k] for swiglu workloads; x [m, k] for
    plain workloads."""
    m = w.m if m is None else m
    g = _gen(w.seed, device)
    if w.kind == "plain":
        return {"x": _bf16(torch.randn(m, w.k, generator=g, device=device, dtype=torch.float32))}
    if w.kind == "swiglu":
        gate = torch.randn(m, w.k, generator=g, device=device, dtype=torch.float32)
        up = torch.randn(m, w.k, generator=g, device=device, dtype=torch.float32)
        return {"gate": _bf16(gate), "up": _bf16(up)}
    z = torch.randn(m, w.k, generator=g, device=device, dtype=torch.float32)
    if w.rms_rows:
        z = z / z.square().mean(dim=1, keepdim=True).sqrt()
    if w.outlier_frac > 0:
        pick = torch.rand(m, w.k, generator=g, device=device) < w.outlier_frac
        big = torch.randn(m, w.k, generator=g, device=device) * w.outlier_std
        z = torch.where(pick, big, z)
    nseg = len(w.seg_off) - 1
    gm = _gen(w.seed + 1000, device)
    shift = torch.randn(nseg, w.k, generator=gm, device=device) * w.mod_std
    scale = torch.randn(nseg, w.k, generator=gm, device=device) * w.mod_std
    return {"x": _bf16(z), "shift": _bf16(shift), "scale": _bf16(scale)}


def seg_offsets(w: Workload, m: int | None = None) -> list:
    """Segment row offsets, with the last one clipped to m rows."""
    m = w.m if m is None else m
    if not w.seg_off:
        return [0, m]
    offs = [min(o, m) for o in w.seg_off]
    offs[-1] = m
    return offs


def weights(w: Workload, device="cpu") -> dict:
    """Packed NVFP4 weight [n, k]: random E2M1 byte pairs, random E4M3 codes in
    [sf_code_lo, sf_code_hi] as a LOGICAL [ceil128(n), k/16] matrix (rows past
    n are zero), and the FP32 weight tensor scale."""
    g = _gen(w.seed + 100, device)
    q = torch.randint(0, 256, (w.n, w.k // 2), generator=g, device=device, dtype=torch.int32).to(torch.uint8)
    rows = -(-w.n // 128) * 128
    sf = torch.zeros(rows, w.k // 16, dtype=torch.uint8, device=device)
    sf[: w.n] = torch.randint(w.sf_code_lo, w.sf_code_hi + 1, (w.n, w.k // 16), generator=g,
                              device=device, dtype=torch.int32).to(torch.uint8)
    return {"q": q, "sf": sf, "ts": float(w.w_ts)}
