"""The C ABI used from plain C: tests/cuda/c_abi_step.c links libob.so and
the CUDA runtime (no Python, no torch), runs 2 warmup and 3 compressed
1-bit Adam steps and compares parameters, server sign words and scales
bit for bit with the oracle's C functions after every step."""
import os
import subprocess

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_program_drives_the_abi(tmp_path):
    from momentum_compression_gb300 import _build
    import oracle.build as obuild
    lib_dir = os.path.dirname(_build.build())
    ora_dir = os.path.dirname(obuild.build())
    exe = str(tmp_path / "c_abi_step")
    subprocess.run(["nvcc", "-O2", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "cuda", "c_abi_step.c"), "-o", exe,
                    "-L", lib_dir, "-lob", "-L", ora_dir, "-loracle",
                    "-Xlinker", f"-rpath,{lib_dir}:{ora_dir}"], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c abi ok" in r.stdout
