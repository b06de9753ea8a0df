"""Every ob_* call opens one NVTX range named after it and closes it before
returning, so the library's calls show up by name on a profiler's timeline
(tracing).  Checked on the CPU: a child process loads libob.so with a small
NVTX injection library (tests/cuda/nvtx_recorder.c, loaded through
NVTX_INJECTION64_PATH) that records every push and pop, and makes calls
that need no GPU -- layout and workspace queries, and calls that are
rejected on the host before any CUDA call."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA_INC = "/usr/local/cuda/include"

CHILD = r'''
import ctypes as ct, sys
sys.path.insert(0, sys.argv[1])
import momentum_compression_gb300 as ob
L = ob.lib()
ctx = ob.ob_init(100_000, 4, 8192)
ob.ob_get_layout(ctx)
ob.ob_workspace_bytes(ctx)
for call in (lambda: ob.ob_compress(ctx, [None] * 4, None, [None] * 4, None, None, stream=0),
             lambda: ob.ob_server_reduce(ctx, None, None, None, None, None, stream=0),
             lambda: ob.ob_adam_step(ctx, None, None, None, None, None, stream=0),
             lambda: ob.ob_error_norm(ctx, [None] * 4, None, None, None, None, None, None,
                                      stream=0),
             lambda: ob.ob_quant_int8(None, None, None, 1, 0, n=0, stream=0),
             lambda: ob.ob_compress_noalloc(ctx, [None] * 4, None, [None] * 4, None, None,
                                            stream=0),
             lambda: ob.ob_reset_errors_rank(ctx, 9, None, None, None, None, None, None,
                                             stream=0)):
    try:
        call()
    except ob.OBError:
        pass
    else:
        raise SystemExit("a call that must fail on the host succeeded")
ob.ob_destroy(ctx)
print("child ok")
'''


def test_every_call_opens_and_closes_a_named_range(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None or not os.path.exists(os.path.join(CUDA_INC, "nvtx3", "nvToolsExt.h")):
        pytest.skip("needs a C compiler and the CUDA toolkit's NVTX headers")
    from momentum_compression_gb300 import _build
    _build.build()
    tool = str(tmp_path / "nvtx_recorder.so")
    subprocess.run([cc, "-std=c11", "-Wall", "-Werror", "-shared", "-fPIC", f"-I{CUDA_INC}",
                    "-o", tool, os.path.join(ROOT, "tests", "cuda", "nvtx_recorder.c")],
                   check=True)
    log = tmp_path / "ranges.log"
    env = dict(os.environ, NVTX_INJECTION64_PATH=tool, OB_NVTX_LOG=str(log))
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0 and "child ok" in r.stdout, r.stderr
    events = log.read_text().split("\n")[:-1]
    pushes = [e.split(" ", 1)[1] for e in events if e.startswith("push ")]
    # the binding reads ob_last_error after every rejected call
    failing = ["ob_compress", "ob_server_reduce", "ob_adam_step", "ob_error_norm",
               "ob_quant_int8", "ob_compress_noalloc", "ob_reset_errors_rank"]
    want = ["ob_init", "ob_get_layout", "ob_workspace_bytes"]
    for name in failing:
        want += [name, "ob_last_error"]
    want.append("ob_destroy")
    assert pushes == want, pushes
    depth = 0
    for e in events:
        depth += 1 if e.startswith("push ") else -1
        assert depth in (0, 1), "ranges must not be left open or nested here"
    assert depth == 0


def test_every_entry_point_opens_its_range_first():
    """Source check for the calls the child above cannot reach without a
    GPU: the body of every exported ob_* function starts with OB_TRACE()."""
    import re
    import momentum_compression_gb300 as ob
    csrc = os.path.join(ROOT, "momentum_compression_gb300", "csrc")
    src = "".join(open(os.path.join(csrc, f)).read() for f in sorted(os.listdir(csrc))
                  if f.endswith(".cu"))
    for name in ob.EXPORTS:
        m = re.search(r"\b" + name + r"\s*\([^;{]*\)\s*\{", src)
        assert m, f"{name}: no definition under csrc/"
        first = src[m.end():].lstrip().split("\n", 1)[0].strip()
        assert first == "OB_TRACE();", f"{name} starts with {first!r}"
