"""Host check of the division-free quotient the pack kernels use for the
block scales and the E2M1 codes.

With r = RN(1/b), q = RN(a r), e = RN(q b - a) and q' = RN(q - e r) (both
fused multiply-adds, IEEE single precision), q' equals the IEEE quotient
RN(a / b) -- the residual correction of Markstein's division.  The kernels
rely on it for every bf16 a and every f32 b in the range they apply it to;
`tests/helpers/rcp_quotient_check.c` compares the two for every bf16
significand of a, every third f32 significand of b in [1, 2) and quotients in
[2^-5, 2^5), both signs and signed zeros (power-of-two scaling carries the
result to every exponent where the residual keeps its bits).  A stride of 1
(all 2^23 significands, 1.9e10 cases) also finds no difference; it takes
~2 CPU-minutes.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


SRC = os.path.join(ROOT, "tests", "helpers", "rcp_quotient_check.c")


def _build(tmp_path, src=SRC, name="rcp_quotient_check"):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not found")
    exe = str(tmp_path / name)
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-o", exe, src, "-lm"]
    if subprocess.run(base[:1] + ["-fopenmp"] + base[1:], capture_output=True).returncode != 0:
        subprocess.run(base, check=True, capture_output=True)
    return exe


def test_division_free_quotient_equals_ieee_quotient(tmp_path):
    exe = _build(tmp_path)
    r = subprocess.run([exe, "3"], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    checks, bad = (int(v) for v in r.stdout.split()[1::2])
    assert checks > 6_000_000_000 // 3 and bad == 0


def test_the_check_catches_a_reciprocal_one_ulp_off(tmp_path):
    """The same comparison with r rounded the wrong way (one ulp off) must
    report mismatches (18 in 2e8 cases at this stride): the check can fail,
    and the correctly rounded reciprocal is what the kernels need."""
    text = open(SRC).read()
    assert "const float r = 1.0f / b;" in text
    bad_src = tmp_path / "rcp_off.c"
    bad_src.write_text(text.replace("const float r = 1.0f / b;", "const float r = nextafterf(1.0f / b, 0.0f);"))
    exe = _build(tmp_path, str(bad_src), "rcp_off")
    r = subprocess.run([exe, "97"], capture_output=True, text=True, timeout=600)
    assert r.returncode == 1 and int(r.stdout.split()[3]) > 0
