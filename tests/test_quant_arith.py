"""The GPU quantizer computes d = amax/127 and 1/d without the division
routines (fma-based methods whose branch-free form lets the blocks of a batch
overlap).  The quantization rule needs both correctly rounded, since their
bits decide the quants.  This test compiles a host restatement of the two
methods (tests/native/quant_arith.c: IEEE float multiplies and fmas only, so
host and device compute the same bits) and checks it against IEEE division
over every significand at many exponents, every subnormal and the special
values.  The device code itself is checked over every significand of amax in
the GPU quantization sweep (test_gpu_quant_sweep.py)."""
import os
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def test_division_free_quotient_and_reciprocal_are_correctly_rounded(tmp_path):
    exe = str(tmp_path / "quant_arith")
    src = os.path.join(HERE, "native", "quant_arith.c")
    try:
        subprocess.run(["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math", src,
                        "-o", exe, "-lm"], check=True, capture_output=True, text=True)
    except FileNotFoundError:
        pytest.skip("no host C compiler")
    r = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    lines = r.stdout.strip().splitlines()
    assert len(lines) == 3 and all(" 0 of " in ln for ln in lines), r.stdout
