"""The oracle's NVFP4 byte conventions against a library routine: nibble order
(element 2i in the low nibble) and the 128x4-atom scale layout (reading R12)
are the public VEC16_UE4M3 convention that cuBLASLt's block-scaled GEMM reads.
The oracle packs activations; cuBLASLt multiplies the oracle's bytes (a
separate program, dit_modulate_absmax_gb300/cublaslt_ref.cu); its output must
lie within the GEMM tolerance of the oracle's FP64 sums.  A swapped nibble
order or a mis-placed scale would put most outputs far outside it.  None of
the library's kernels is involved."""
import subprocess

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu


def test_cublaslt_reads_the_oracles_packed_operands_as_intended(tmp_path):
    from dit_modulate_absmax_gb300 import compare_cublaslt
    exe = compare_cublaslt.build_ref()
    rng = np.random.default_rng(81)
    m, m_pad, n, k = 300, 320, 256, 512
    x = rng.standard_normal((m, k)).astype(np.float32)
    x[5, :16] = 0.0                                       # an all-zero block
    xb = (x.view(np.uint32) + 0x7FFF + ((x.view(np.uint32) >> 16) & 1)) >> 16   # fp32 -> bf16 (RNE) patterns
    ts_a, q_a, sf_a, _ = oracle.plain_producer(xb.astype(np.uint16), m_pad)
    q_b = rng.integers(0, 256, size=(n, k // 2), dtype=np.uint8)
    sf_b = rng.integers(0x30, 0x48, size=(n, k // 16)).astype(np.uint8)
    ts_b = 2.0 ** -3
    m128 = -(-m // 128) * 128
    aq = np.zeros((m128, k // 2), dtype=np.uint8)
    aq[:m_pad] = q_a
    for name, arr in (("aq.bin", aq), ("asf.bin", oracle.swizzle_sf(sf_a)), ("bq.bin", q_b),
                      ("bsf.bin", oracle.swizzle_sf(sf_b))):
        arr.tofile(tmp_path / name)
    alpha = float(np.float32(ts_a) * np.float32(ts_b))
    out = tmp_path / "c.bin"
    r = subprocess.run([exe, str(tmp_path), str(m), str(n), str(k), "1", repr(alpha), str(out)],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    C = np.fromfile(out, dtype=np.uint16).reshape(m, n)
    R, S = oracle.gemm_reference(q_a, sf_a, ts_a, q_b, sf_b, ts_b, k, rows=np.arange(m))
    ok, err, tol = oracle.gemm_check(C, R, S)
    assert ok.all(), f"{int((~ok).sum())} of {ok.size} outputs outside tolerance (max err/tol {float((err / tol).max()):.3g})"
    assert np.abs(R).max() > 1.0                          # the products are not trivially zero
