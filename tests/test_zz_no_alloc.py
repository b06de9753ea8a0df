"""ob_compress_noalloc, the compression entry point for callers that cannot
allocate device memory (it uses the library's static scratch array
instead of a caller-provided workspace), and ob_noalloc_device_error, the
reader of that array's error word.

Checked here: two calls in a row against the oracle and against
ob_compress, bit for bit; that calls after the first change neither the
device's free memory nor torch's allocator counters; that the error word
reads 0 after normal calls; replays of a captured call; and the exact size
rule.

Kept in a file that pytest collects last, so that a run stopping at the
first failure has already run every other test.  It passes alone in a
fresh process as well as after the other tests.
"""
import gc

import pytest
import torch

import momentum_compression_gb300 as ob
import oracle as O
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


def _ws_ctx(n, W, chunk, grad_dtype):
    ctx = ob.ob_init(n, W, chunk, grad_dtype=grad_dtype)
    nb = ob.ob_workspace_bytes(ctx)
    ws = torch.zeros((nb + 255) // 4, device="cuda")
    ob.ob_set_workspace(ctx, ws, nb)
    return ctx, ws


CASES = [
    (1 << 20, 4, 1 << 18, ob.OB_GRAD_F32),
    (300_001, 8, 1 << 14, ob.OB_GRAD_BF16),
]


@pytest.mark.parametrize("n,W,chunk,grad_dtype", CASES)
def test_noalloc_matches_oracle_and_compress_twice(n, W, chunk, grad_dtype):
    """Two calls in a row (the second decodes the first's deferred errors):
    sign words, scales and stored compensated values equal the oracle's and
    ob_compress's, bit for bit -- the tolerance of every single-kernel
    parity test here."""
    ctx_ws, ws = _ws_ctx(n, W, chunk, grad_dtype)
    lay = ob.ob_get_layout(ctx_ws)
    ctx_na = ob.ob_init(n, W, chunk, grad_dtype=grad_dtype)  # no workspace at all
    words, nc = lay["words_per_worker"], lay["n_chunks"]
    olay = O.Layout(n, W, 4096, chunk)
    assert olay.n_pad == lay["n_pad"]

    grads, m, err = _buffers(lay, W, n, grad_dtype, seed=11)
    # the oracle's state: the same true errors (scales start at 0, so the
    # deferred values decode to themselves)
    o_e = [host(e).copy() for e in err]
    o_m = host(m).copy()
    err_a = [e.clone() for e in err]
    err_b = [e.clone() for e in err]
    bits_a = torch.zeros((W, words), dtype=torch.int32, device="cuda")
    bits_b = torch.zeros_like(bits_a)
    sc_a = torch.zeros((W, nc), device="cuda")
    sc_b = torch.zeros_like(sc_a)
    for call in range(2):
        if call == 1:
            grads, _, _ = _buffers(lay, W, n, grad_dtype, seed=12)
        ob.ob_compress(ctx_ws, grads, m, err_a, bits_a, sc_a)
        ob.ob_compress_noalloc(ctx_na, grads, m, err_b, bits_b, sc_b)
        torch.cuda.synchronize()
        assert ob.ob_noalloc_device_error() == 0
        got_bits, got_sc = host(bits_b), host(sc_b)
        for w in range(W):
            ob_bits, ob_sc, ob_x = O.compress_worker(olay, host(grads[w].float()), o_m, o_e[w],
                                                     0.9)
            what = f"worker {w}, call {call}"
            assert_bits_equal(got_bits[w, :olay.words], ob_bits, f"sign words vs oracle, {what}")
            assert_bits_equal(got_sc[w], ob_sc, f"scales vs oracle, {what}")
            assert_bits_equal(host(err_b[w]), ob_x, f"stored x vs oracle, {what}")
            assert_bits_equal(host(err_b[w]), host(err_a[w]), f"stored x vs ob_compress, {what}")
        assert_bits_equal(got_bits, host(bits_a), f"sign words vs ob_compress, call {call}")
        assert_bits_equal(got_sc, host(sc_a), f"scales vs ob_compress, call {call}")
    ob.ob_destroy(ctx_ws)
    ob.ob_destroy(ctx_na)


def test_noalloc_allocates_nothing():
    """After the first call (which looks up the array's address), calls
    leave the device's free memory and torch's allocator counters as they
    were."""
    n, W, chunk, gd = CASES[0]
    ctx = ob.ob_init(n, W, chunk, grad_dtype=gd)
    lay = ob.ob_get_layout(ctx)
    grads, m, err = _buffers(lay, W, n, gd, seed=21)
    bits = torch.zeros((W, lay["words_per_worker"]), dtype=torch.int32, device="cuda")
    sc = torch.zeros((W, lay["n_chunks"]), device="cuda")
    ob.ob_compress_noalloc(ctx, grads, m, err, bits, sc)
    assert ob.ob_noalloc_device_error() == 0  # synchronises
    # tensors left by earlier tests are freed now, not during the calls
    gc.collect()
    torch.cuda.synchronize()
    stats0 = torch.cuda.memory_stats()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(5):
        ob.ob_compress_noalloc(ctx, grads, m, err, bits, sc)
    assert ob.ob_noalloc_device_error() == 0
    free1, _ = torch.cuda.mem_get_info()
    stats1 = torch.cuda.memory_stats()
    assert free1 == free0, f"device free memory changed by {free1 - free0} bytes"
    # counters that only grow when something is allocated: torch's
    # allocations and its cudaMalloc'd segments, and the memory it holds
    for k in ("allocation.all.allocated", "segment.all.allocated", "reserved_bytes.all.current"):
        assert stats1.get(k, 0) == stats0.get(k, 0), k
    ob.ob_destroy(ctx)


def test_noalloc_graph_replays_match_compress():
    """One eager call, then the call captured in a CUDA graph and replayed
    twice with new gradients: bit for bit ob_compress's results."""
    n, W, chunk, gd = CASES[1]
    ctx_ws, ws = _ws_ctx(n, W, chunk, gd)
    lay = ob.ob_get_layout(ctx_ws)
    ctx_na = ob.ob_init(n, W, chunk, grad_dtype=gd)
    grads, m, err = _buffers(lay, W, n, gd, seed=31)
    err_a = [e.clone() for e in err]
    err_b = [e.clone() for e in err]
    bits_a = torch.zeros((W, lay["words_per_worker"]), dtype=torch.int32, device="cuda")
    bits_b = torch.zeros_like(bits_a)
    sc_a = torch.zeros((W, lay["n_chunks"]), device="cuda")
    sc_b = torch.zeros_like(sc_a)
    ob.ob_compress(ctx_ws, grads, m, err_a, bits_a, sc_a)
    ob.ob_compress_noalloc(ctx_na, grads, m, err_b, bits_b, sc_b)  # eager, first
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        ob.ob_compress_noalloc(ctx_na, grads, m, err_b, bits_b, sc_b)
    for rep in range(2):
        new, _, _ = _buffers(lay, W, n, gd, seed=32 + rep)
        for g, x in zip(grads, new):
            g.copy_(x)
        ob.ob_compress(ctx_ws, grads, m, err_a, bits_a, sc_a)
        graph.replay()
        torch.cuda.synchronize()
        assert_bits_equal(host(bits_b), host(bits_a), f"sign words, replay {rep}")
        assert_bits_equal(host(sc_b), host(sc_a), f"scales, replay {rep}")
        for w in range(W):
            assert_bits_equal(host(err_b[w]), host(err_a[w]), f"x of worker {w}, replay {rep}")
    assert ob.ob_noalloc_device_error() == 0
    del graph
    ob.ob_destroy(ctx_ws)
    ob.ob_destroy(ctx_na)


def test_noalloc_size_rule():
    """A layout is accepted exactly when W * n_chunks * ceil(chunk/4096) * 4
    <= OB_NOALLOC_SCRATCH_BYTES - 256.  At W = 8 with chunk 4096 that allows
    16383 chunks per partition; 16384 are rejected before any launch, with
    a message stating both sizes.  (The layout at the limit is not launched
    here: its buffers would need 34 GB.)"""
    limit = ob.OB_NOALLOC_SCRATCH_BYTES - 256
    dummy = torch.zeros(16, device="cuda")
    # 16384 chunks of 4096 per partition: 8 * (8 * 16384) * 1 * 4 = limit + 256
    ctx = ob.ob_init(8 * 16384 * 4096, 8, 4096)
    lay = ob.ob_get_layout(ctx)
    assert 8 * lay["n_chunks"] * 4 == limit + 256
    with pytest.raises(ob.OBError) as ei:
        ob.ob_compress_noalloc(ctx, [dummy] * 8, dummy, [dummy] * 8, dummy, dummy)
    assert ei.value.status == ob.OB_ERR_UNSUPPORTED
    assert f"needs {limit + 256} bytes" in ob.ob_last_error(ctx)
    assert f"holds {limit}" in ob.ob_last_error(ctx)
    ob.ob_destroy(ctx)
    # 2^30 elements at W = 8 need about 8 MiB of per-tile totals
    ctx = ob.ob_init(1 << 30, 8, 1 << 20)
    with pytest.raises(ob.OBError) as ei:
        ob.ob_compress_noalloc(ctx, [dummy] * 8, dummy, [dummy] * 8, dummy, dummy)
    assert ei.value.status == ob.OB_ERR_UNSUPPORTED
    assert "static scratch" in ob.ob_last_error(ctx)
    ob.ob_destroy(ctx)
