"""Failure detection on the GPU without a fault: the bounded mbarrier wait of
the pipelined kernels gives up after its limit, records an error code the
host can read, and returns; the context stays usable.

The wait is driven to its limit the way a lost copy would: by waiting on a
barrier phase that nothing completes (a flag nothing sets)."""
import ctypes as ct
import os
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "momentum_compression_gb300", "csrc")


@pytest.fixture(scope="module")
def lib(tmp_path_factory):
    out = str(tmp_path_factory.mktemp("waits") / "libwaits.so")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-shared",
                    "-Xcompiler", "-fPIC", f"-I{CSRC}", "-o", out,
                    os.path.join(HERE, "cuda", "wait_selftest.cu")], check=True)
    L = ct.CDLL(out)
    L.wait_selftest.argtypes = [ct.c_void_p, ct.c_longlong, ct.c_int, ct.c_void_p, ct.c_void_p]
    return L


def _run(lib, limit, arrive_first):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    res = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    cyc = torch.zeros(1, dtype=torch.int64, device="cuda")
    assert lib.wait_selftest(err.data_ptr(), limit, arrive_first, res.data_ptr(),
                             cyc.data_ptr()) == 0
    return int(err.item()), int(res.item()), int(cyc.item())


def test_wait_on_a_phase_nothing_completes_times_out(lib):
    limit = 2_000_000  # about a millisecond
    err, res, cyc = _run(lib, limit, arrive_first=0)
    assert res == 0, "the wait must give up"
    assert err == 1, "and record the consumer-wait code"
    assert limit < cyc < 50 * limit
    # the context is still usable afterwards
    x = torch.arange(10, device="cuda")
    assert int(x.sum().item()) == 45


def test_wait_on_a_completed_phase_returns_at_once(lib):
    err, res, cyc = _run(lib, 2_000_000, arrive_first=1)
    assert res == 1 and err == 0
    assert cyc < 2_000_000
