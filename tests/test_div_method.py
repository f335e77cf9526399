"""The write kernel divides by a per-head scale with a precomputed reciprocal
and one fused residual correction instead of a full IEEE divide per element.
This checks, exhaustively over every bf16 significand and every binary32
divisor significand (both in [1, 2), which fixes the rounding of every
normal quotient), that the method returns the IEEE binary32 quotient."""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))


def test_reciprocal_correction_is_exact(tmp_path):
    exe = tmp_path / "div_check"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off", "-fopenmp",
                    os.path.join(HERE, "csrc", "div_check.c"), "-o", str(exe), "-lm"], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.strip()
    assert out == "0", f"{out} significand pairs differ from IEEE division"
