"""The C ABI used from plain C: the programs under tests/cuda link libob.so
and the CUDA runtime (no Python, no torch) and compare with the oracle's C
functions bit for bit after every step.  c_abi_step.c: 2 warmup and 3
compressed 1-bit Adam steps.  c_abi_lamb_signm.c: 2 warmup and 4
compressed 1-bit LAMB steps over three layers, the last 3 with the
momentum in sign form and the server output double-buffered
(ob_step_db).  c_abi_mixed.c: a 1-bit, a 2-bit and an FP16 group over 7
compressed steps, with the periodic reset, the FP16 send period and the
per-width key taken from the library (ob_plan_step, ob_codec_step)."""
import os
import subprocess

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("prog,ok", [("c_abi_step", "c abi ok"),
                                     ("c_abi_lamb_signm", "c abi lamb ok"),
                                     ("c_abi_mixed", "c abi mixed ok")])
def test_c_program_drives_the_abi(tmp_path, prog, ok):
    from momentum_compression_gb300 import _build
    import oracle.build as obuild
    lib_dir = os.path.dirname(_build.build())
    ora_dir = os.path.dirname(obuild.build())
    exe = str(tmp_path / prog)
    subprocess.run(["nvcc", "-O2", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "cuda", prog + ".c"), "-o", exe,
                    "-L", lib_dir, "-lob", "-L", ora_dir, "-loracle",
                    "-Xlinker", f"-rpath,{lib_dir}:{ora_dir}"], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert ok in r.stdout
