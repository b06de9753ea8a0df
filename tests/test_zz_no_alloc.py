"""ob_compress_noalloc, the compression entry point for callers that cannot
allocate device memory (it uses the library's static scratch array
instead of a caller-provided workspace), against ob_compress.

Kept in a file that pytest collects last, so that a run stopping at the
first failure has already run every other test.  It passes alone in a
fresh process as well as after the other tests.
"""
import numpy as np
import pytest
import torch

import momentum_compression_gb300 as ob
from helpers import assert_bits_equal, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)
    from momentum_compression_gb300 import _build
    _build.build()


def _buffers(lay, W, n, grad_dtype, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    n_pad = lay["n_pad"]

    def vec(scale):
        t = torch.zeros(n_pad, device="cuda")
        t[:n] = torch.randn(n, generator=g, device="cuda") * scale
        return t

    grads = [vec(1e-3).to(torch.bfloat16 if grad_dtype else torch.float32) for _ in range(W)]
    return grads, vec(1e-3), [vec(1e-4) for _ in range(W)]


@pytest.mark.parametrize("n,W,chunk,grad_dtype", [
    (1 << 20, 4, 1 << 18, ob.OB_GRAD_F32),
    (300_001, 8, 1 << 14, ob.OB_GRAD_BF16),
])
def test_noalloc_matches_compress_twice(n, W, chunk, grad_dtype):
    # reference: the existing entry point with a workspace
    ctx_ws = ob.ob_init(n, W, chunk, grad_dtype=grad_dtype)
    lay = ob.ob_get_layout(ctx_ws)
    nb = ob.ob_workspace_bytes(ctx_ws)
    ws = torch.zeros((nb + 255) // 4, device="cuda")
    ob.ob_set_workspace(ctx_ws, ws, nb)
    # the new entry point: a ctx with no workspace at all
    ctx_na = ob.ob_init(n, W, chunk, grad_dtype=grad_dtype)
    words, nc = lay["words_per_worker"], lay["n_chunks"]

    grads, m, err = _buffers(lay, W, n, grad_dtype, seed=11)
    err_a = [e.clone() for e in err]
    err_b = [e.clone() for e in err]
    bits_a = torch.zeros((W, words), dtype=torch.int32, device="cuda")
    bits_b = torch.zeros_like(bits_a)
    sc_a = torch.zeros((W, nc), device="cuda")
    sc_b = torch.zeros_like(sc_a)
    for call in range(2):  # two calls in a row: the second reads the first's state
        if call == 1:
            grads, _, _ = _buffers(lay, W, n, grad_dtype, seed=12)
        ob.ob_compress(ctx_ws, grads, m, err_a, bits_a, sc_a)
        ob.ob_compress_noalloc(ctx_na, grads, m, err_b, bits_b, sc_b)
        torch.cuda.synchronize()
        # bit-exact, the tolerance of every single-kernel parity test here
        assert_bits_equal(host(bits_b), host(bits_a), f"sign words, call {call}")
        assert_bits_equal(host(sc_b), host(sc_a), f"scales, call {call}")
        for w in range(W):
            assert_bits_equal(host(err_b[w]), host(err_a[w]), f"errors of worker {w}, call {call}")
    ob.ob_destroy(ctx_ws)
    ob.ob_destroy(ctx_na)


def test_noalloc_rejects_layouts_beyond_its_scratch():
    # 2^30 elements at W = 8 need about 8 MiB of per-tile totals
    ctx = ob.ob_init(1 << 30, 8, 1 << 20)
    dummy = torch.zeros(16, device="cuda")
    with pytest.raises(ob.OBError) as ei:
        ob.ob_compress_noalloc(ctx, [dummy] * 8, dummy, [dummy] * 8, dummy, dummy)
    assert ei.value.status == ob.OB_ERR_UNSUPPORTED
    assert "static scratch" in ob.ob_last_error(ctx)
    ob.ob_destroy(ctx)
