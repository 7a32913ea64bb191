"""The oracle's fp32 -> bf16 rounding on all 2^32 fp32 bit patterns, against
a second formulation written independently in tests/native/bf16_exhaustive.c:
the nearer of the two bf16 neighbours by exact distance in double, ties to the
even one, overflow to infinity; NaN in gives NaN of the same sign.  bf16 rounding
decides every bf16 result (FSDP collectives 101, "Why backward needs a
different collective": bf16 gradients are reduced and rounded to bf16)."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def test_bf16_rounding_every_pattern(oracle_mod, tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("needs a C compiler")
    exe = tmp_path / "bf16_exhaustive"
    subprocess.run([cc, "-O2", "-std=c11", "-pthread", "-o", str(exe),
                    os.path.join(HERE, "native", "bf16_exhaustive.c"), "-ldl", "-lm"], check=True)
    lib = oracle_mod.build()
    threads = max(1, min(64, os.cpu_count() or 1))
    p = subprocess.run([str(exe), lib, str(threads)], capture_output=True, text=True, timeout=900)
    assert p.returncode == 0 and p.stdout.strip() == "mismatches 0", p.stdout + p.stderr
