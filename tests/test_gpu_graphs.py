"""CUDA graphs and streams.  A compressed step captured in a CUDA graph and
replayed gives the same bits as the same steps called eagerly (1-bit Adam
with the momentum in sign form, 1-bit LAMB with a dense momentum and with
the momentum in sign form, whose two server buffers alternate between two
graphs): the library's calls
allocate nothing and take every per-step quantity from device memory, so a
replay is the step itself.  Two contexts stepped concurrently on two
streams are independent."""
import numpy as np
import pytest
import torch

import momentum_compression_gb300 as ob
from helpers import assert_bits_equal, host

pytestmark = pytest.mark.gpu

HP = dict(b1=0.9, b2=0.999, eps=1e-8, lr=1e-4)


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)
    from momentum_compression_gb300 import _build
    _build.build()


def _make(lamb, seed, sm=None):
    n, W = 300_001, 4
    off = [0, 1000, 70_000, 250_000, n] if lamb else None
    hp = dict(HP, **(dict(r_thr=0.1, r_min=0.5, r_max=4.0, c_min=0.01, c_max=10.0)
                     if lamb else {}))
    opt = ob.OneBitOptimizer(n, W, 1 << 16, 4096, "f32", off, lamb=lamb,
                             sign_momentum=(not lamb) if sm is None else sm, **hp)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    opt.p[:n] = torch.randn(n, generator=gen, device="cuda") * 0.02
    return opt, n, W


def _grads(n_pad, n, W, step):
    gen = torch.Generator(device="cuda")
    gen.manual_seed(1000 + step)
    out = []
    for _ in range(W):
        g = torch.zeros(n_pad, device="cuda")
        g[:n] = torch.randn(n, generator=gen, device="cuda") * 1e-3
        out.append(g)
    return out


@pytest.mark.parametrize("lamb,sm", [(False, True), (True, False), (True, True)])
def test_graph_replay_matches_eager_steps(lamb, sm):
    a, n, W = _make(lamb, 1, sm)
    b, _, _ = _make(lamb, 1, sm)
    for opt in (a, b):
        for t in range(3):
            opt.warmup_step(_grads(opt.n_pad, n, W, t))
        opt.begin_compression()
        opt.compressed_step(_grads(opt.n_pad, n, W, 3))
    bufs = [torch.zeros(b.n_pad, device="cuda") for _ in range(W)]
    graph = b.capture_step(bufs)
    for t in range(4, 10):
        g = _grads(a.n_pad, n, W, t)
        a.compressed_step(g)
        for dst, src in zip(bufs, g):
            dst.copy_(src)
        graph.replay()
        torch.cuda.synchronize()
        assert_bits_equal(host(b.p), host(a.p), f"p after step {t}")
        assert_bits_equal(host(b.sbits), host(a.sbits), f"sbits after step {t}")
        assert_bits_equal(host(b.sscales), host(a.sscales), f"sscales after step {t}")
        assert_bits_equal(host(b.err_s), host(a.err_s), f"e_s after step {t}")
        if lamb:
            assert_bits_equal(host(b.ls.c_t), host(a.ls.c_t), f"c_t after step {t}")
    a.close()
    b.close()


def test_replay_refuses_a_changed_momentum_form():
    """A graph captured with the momentum in sign form does not replay once
    materialize_m has made it dense again."""
    opt, n, W = _make(True, 3, sm=True)
    for t in range(2):
        opt.warmup_step(_grads(opt.n_pad, n, W, t))
    opt.begin_compression()
    opt.compressed_step(_grads(opt.n_pad, n, W, 2))
    bufs = _grads(opt.n_pad, n, W, 3)  # the graph reads these buffers
    graph = opt.capture_step(bufs)
    graph.replay()
    opt.materialize_m()
    with pytest.raises(RuntimeError):
        graph.replay()
    torch.cuda.synchronize()
    opt.close()


def test_capture_refuses_host_schedules():
    opt, n, W = _make(False, 2)
    opt.begin_compression()
    with pytest.raises(ValueError):
        opt.capture_step(_grads(opt.n_pad, n, W, 0))   # momentum still dense
    opt.close()


def test_two_contexts_on_two_streams_are_independent():
    """Two jobs (own ctx, workspace and buffers) stepped concurrently on two
    streams give the same bits as the same jobs stepped one after the
    other: nothing in the library is shared between contexts."""
    runs = []
    for concurrent in (False, True):
        jobs = [_make(False, 10 + j) for j in range(2)]
        streams = [torch.cuda.Stream() for _ in range(2)]
        torch.cuda.synchronize()  # the initial parameters were written on the default stream
        for (opt, n, W), s in zip(jobs, streams):
            with torch.cuda.stream(s):
                for t in range(2):
                    opt.warmup_step(_grads(opt.n_pad, n, W, t), stream=s)
                opt.begin_compression(stream=s)
        torch.cuda.synchronize()
        grads = [[_grads(opt.n_pad, n, W, 10 * j + t) for t in range(4)]
                 for j, (opt, n, W) in enumerate(jobs)]
        torch.cuda.synchronize()
        if concurrent:
            for t in range(4):
                for j, ((opt, n, W), s) in enumerate(zip(jobs, streams)):
                    opt.compressed_step(grads[j][t], stream=s)
        else:
            for j, ((opt, n, W), s) in enumerate(zip(jobs, streams)):
                for t in range(4):
                    opt.compressed_step(grads[j][t], stream=s)
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        runs.append([(host(opt.p).copy(), host(opt.sbits).copy()) for opt, _, _ in jobs])
        for opt, _, _ in jobs:
            assert ob.ob_device_error(opt.ctx) == 0
            opt.close()
    for (p0, s0), (p1, s1) in zip(runs[0], runs[1]):
        assert_bits_equal(p1, p0, "p")
        assert_bits_equal(s1, s0, "sbits")
