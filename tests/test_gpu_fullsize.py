"""Parity at the workloads' full sizes, in the launch configuration bench.py
times (the same OneBitOptimizer calls, grids sized by the library).

The 1-bit Adam step is chunk-local: every output element depends only on
the inputs of its own chunk (the chunk's scale, its W workers' signs, the
server's error), and Adam's warmup step is elementwise.  So the Adam tests
run the full-size steps on the GPU and the oracle on a few sampled chunks
-- the first, one in the middle, the last real one (with the padding tail)
and the short last chunk of a partition -- as problems of their own, over
the configurations' own step counts, and compare them element by element.
1-bit LAMB's per-layer coefficient needs whole layers, so its multi-step
test runs the oracle on the whole buffer, split over the partitions on a
thread pool (tests/oracle_parallel.py).

Inputs are drawn on the GPU by torch's seeded generator with the synth
recipe's distributions (host generation of billions of values would take
minutes); the slices the oracle needs are copied to the host before each
step.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import momentum_compression_gb300 as ob
import oracle as O
import oracle_parallel as OP
import synth
from helpers import assert_bits_equal, assert_close, host

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

f32 = np.float32


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)
    from momentum_compression_gb300 import _build
    _build.build()
    yield
    torch.cuda.empty_cache()


def _free_bytes():
    free, _ = torch.cuda.mem_get_info()
    return free


def _gen(seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return g


def _std_vector(wl, n_pad):
    std = torch.zeros(n_pad, device="cuda")
    if wl.tensors is None:
        std[: wl.n] = wl.flat_std
    else:
        sizes = torch.tensor([s for _, s, _ in wl.tensors], device="cuda")
        std[: wl.n] = torch.repeat_interleave(
            torch.tensor(wl.layer_std, dtype=torch.float32, device="cuda"), sizes)
    return std


def _fill_state(opt, wl, seed):
    """Compressed-phase state drawn directly: m, e, e_s ~ N(0, 1e-3 / 1e-4),
    v ~ |N(0, 1e-6)| + 1e-12, p ~ N(0, 0.02); padding stays 0."""
    n = wl.n
    g = _gen(seed)
    opt.m[:n] = torch.randn(n, generator=g, device="cuda") * 1e-3
    opt.v[:n] = torch.randn(n, generator=g, device="cuda").abs() * 1e-6 + 1e-12
    opt.p[:n] = torch.randn(n, generator=g, device="cuda") * 0.02
    for e in opt.err:
        e[:n] = torch.randn(n, generator=g, device="cuda") * 1e-4
    opt.err_s[:n] = torch.randn(n, generator=g, device="cuda") * 1e-4
    if opt.v_fresh is not None:
        opt.v_fresh.copy_(opt.v)
    # deferred form with zero scales: err holds the true errors
    opt.scales.zero_()
    opt.sscales.zero_()
    opt.bits.zero_()
    opt.sbits.zero_()


def _grads(opt, wl, step, std):
    g = _gen(synth.SEED_BASE + 1000 * step)
    dt = torch.bfloat16 if wl.grad_dtype == "bf16" else torch.float32
    return [(torch.randn(opt.n_pad, generator=g, device="cuda") * std).to(dt) for _ in range(wl.W)]


def _chunks(lay, n):
    P, C, cpp = lay["P"], lay["chunk"], lay["chunks_per_partition"]
    W = lay["W"]
    out = []

    def rng(g):
        j, kc = divmod(g, cpp)
        s = j * P + kc * C
        ln = min(C, P - kc * C)
        return g, s, ln, max(0, min(n - s, ln))

    picks = {0, (W * cpp) // 2, cpp - 1}
    last_real = (n - 1) // P * cpp + ((n - 1) % P) // C
    picks.add(last_real)
    for g in sorted(picks):
        c = rng(g)
        if c[3] > 0:
            out.append(c)
    return out


def _slices(opt, chunks):
    """Host copies of every buffer a chunk's step reads."""
    d = {}
    for g, s, ln, r in chunks:
        d[g] = dict(
            m=host(opt.m[s:s + ln]).copy(), v=host(opt.v[s:s + ln]).copy(),
            p=host(opt.p[s:s + ln]).copy(), e_s=host(opt.err_s[s:s + ln]).copy(),
            e=[host(e[s:s + ln]).copy() for e in opt.err],
            v_fresh=None if opt.v_fresh is None else host(opt.v_fresh[s:s + ln]).copy())
    return d


def _grad_slices(grads, chunks):
    out = {}
    for g, s, ln, r in chunks:
        out[g] = [host(x[s:s + ln].float()).copy() for x in grads]
    return out


class ChunkOracle:
    """The oracle run on one chunk as a problem of its own: a layout with
    n = real elements, alignment = chunk = the chunk's length, so that chunk
    0 is exactly the sampled chunk and every other chunk is padding."""

    def __init__(self, W, s, ln, r, st, layers=None):
        self.W, self.s, self.ln, self.r = W, s, ln, r
        self.lay = O.Layout(r, W, ln, ln)
        assert self.lay.P == ln and self.lay.cpp == 1
        npd = self.lay.n_pad
        self.state = O.State(self.lay, layers, lamb=st["v_fresh"] is not None)
        S = self.state

        def put(dst, src):
            dst[:ln] = src
            dst[r:] = 0

        put(S.m, st["m"])
        put(S.v, st["v"])
        put(S.p, st["p"])
        put(S.e_s, st["e_s"])
        for w in range(W):
            put(S.e[w], st["e"][w])
        if S.v_fresh is not None:
            put(S.v_fresh, st["v_fresh"])
        self.npd = npd

    def grads(self, gs):
        out = []
        for w in range(self.W):
            a = np.zeros(self.npd, f32)
            a[: self.ln] = gs[w]
            a[self.r:] = 0
            out.append(a)
        return out


def _compare_chunk(opt, co, g, what):
    S, s, ln, r = co.state, co.s, co.ln, co.r
    words = ln // 32
    assert_bits_equal(host(opt.sbits[s // 32: s // 32 + words]), S.sbits[:words], f"{what} sbits")
    assert_bits_equal(host(opt.sscales[g]), S.sscales[0], f"{what} sscale")
    for w in range(co.W):
        assert_bits_equal(host(opt.bits[w, s // 32: s // 32 + words]), S.bits[w, :words],
                          f"{what} bits[{w}]")
        assert_bits_equal(host(opt.scales[w, g]), S.scales[w, 0], f"{what} scale[{w}]")
    assert_bits_equal(host(opt.m[s:s + ln]), S.m[:ln], f"{what} m")
    if opt.v_fresh is not None:
        assert_bits_equal(host(opt.v_fresh[s:s + r]), S.v_fresh[:r], f"{what} v_fresh")


def _compare_chunk_errors_and_p(opt, co, what, p_exact=True):
    S, s, ln, r = co.state, co.s, co.ln, co.r
    assert_bits_equal(host(opt.err_s[s:s + ln]), S.e_s[:ln], f"{what} e_s")
    for w in range(co.W):
        assert_bits_equal(host(opt.err[w][s:s + ln]), S.e[w][:ln], f"{what} e[{w}]")
    if p_exact:
        assert_close(host(opt.p[s:s + r]), S.p[:r], f"{what} p")
        assert_bits_equal(host(opt.p[s:s + r]), S.p[:r], f"{what} p")


def _run_adam_fullsize(wl, steps=2, need_bytes=None, sign_momentum=False):
    if need_bytes and _free_bytes() < need_bytes:
        pytest.skip(f"needs {need_bytes / 1e9:.0f} GB of free device memory")
    opt = ob.OneBitOptimizer(wl.n, wl.W, wl.chunk, wl.align, wl.grad_dtype,
                             sign_momentum=sign_momentum, **wl.hp)
    std = _std_vector(wl, opt.n_pad)
    _fill_state(opt, wl, seed=99)
    chunks = _chunks(opt.layout, wl.n)
    st0 = _slices(opt, chunks)
    cos = {g: ChunkOracle(wl.W, s, ln, r, st0[g]) for g, s, ln, r in chunks}
    for t in range(steps):
        grads = _grads(opt, wl, t, std)
        gsl = _grad_slices(grads, chunks)
        opt.compressed_step(grads)
        for g, co in cos.items():
            O.compressed_step(co.state, co.grads(gsl[g]), wl.hp)
        del grads
    torch.cuda.synchronize()
    assert ob.ob_device_error(opt.ctx) == 0
    opt.materialize_m()
    for g, co in cos.items():
        _compare_chunk(opt, co, g, f"chunk {g}")
    opt.materialize_errors()
    torch.cuda.synchronize()
    for g, co in cos.items():
        _compare_chunk_errors_and_p(opt, co, f"chunk {g}")
    opt.close()


@pytest.mark.parametrize("sign_momentum", [False, True])
def test_bert_base_full_size(sign_momentum):
    """109,482,240 parameters (199 tensors), W = 8, chunk 2^20, fp32: the
    workload bench.py times (with the momentum in sign form, as bench.py
    runs it, and dense), 10 compressed steps."""
    _run_adam_fullsize(synth.workload("bert-base"), steps=10, need_bytes=20e9,
                       sign_momentum=sign_momentum)


def _run_adam_from_warmup(wl, warmup, steps, need_bytes, sign_momentum=True):
    """The configuration's own schedule at full size: p0 ~ N(0, 0.02), m =
    v = 0, `warmup` uncompressed steps, the end of warmup, then `steps`
    compressed steps (the momentum in sign form from the second one, as
    bench.py runs it).  The oracle runs the sampled chunks as problems of
    their own (Adam's warmup is elementwise and its compressed step
    chunk-local), on a thread pool.  The sampled server words and scales are
    compared after every compressed step, everything else at the end."""
    if _free_bytes() < need_bytes:
        pytest.skip(f"needs {need_bytes / 1e9:.0f} GB of free device memory")
    opt = ob.OneBitOptimizer(wl.n, wl.W, wl.chunk, wl.align, wl.grad_dtype,
                             sign_momentum=sign_momentum, **wl.hp)
    std = _std_vector(wl, opt.n_pad)
    opt.p[: wl.n] = torch.randn(wl.n, generator=_gen(synth.SEED_BASE + 17), device="cuda") * 0.02
    chunks = _chunks(opt.layout, wl.n)
    st0 = _slices(opt, chunks)
    cos = {g: ChunkOracle(wl.W, s, ln, r, st0[g]) for g, s, ln, r in chunks}
    hp = wl.hp
    with ThreadPoolExecutor(len(cos)) as pool:
        for t in range(warmup):
            grads = _grads(opt, wl, t, std)
            gsl = _grad_slices(grads, chunks)
            opt.warmup_step(grads)
            list(pool.map(lambda g: O.warmup_step(cos[g].lay, cos[g].grads(gsl[g]), 0, hp,
                                                  cos[g].state.m, cos[g].state.v,
                                                  cos[g].state.p), cos))
            del grads
        opt.begin_compression()
        for co in cos.values():
            O.begin_compression(co.state, warmup)
        torch.cuda.synchronize()
        for g, co in cos.items():
            S, a, r = co.state, co.s, co.r
            assert_bits_equal(host(opt.v[a:a + r]), S.v[:r], f"chunk {g}: v after warmup")
            assert_bits_equal(host(opt.p[a:a + r]), S.p[:r], f"chunk {g}: p after warmup")
        for t in range(warmup, warmup + steps):
            grads = _grads(opt, wl, t, std)
            gsl = _grad_slices(grads, chunks)
            opt.compressed_step(grads)
            list(pool.map(lambda g: O.compressed_step(cos[g].state, cos[g].grads(gsl[g]), hp),
                          cos))
            del grads
            torch.cuda.synchronize()
            for g, co in cos.items():
                words = co.ln // 32
                assert_bits_equal(host(opt.sbits[co.s // 32: co.s // 32 + words]),
                                  co.state.sbits[:words], f"chunk {g} sbits at step {t}")
                assert_bits_equal(host(opt.sscales[g]), co.state.sscales[0],
                                  f"chunk {g} sscale at step {t}")
    assert ob.ob_device_error(opt.ctx) == 0
    opt.materialize_m()
    for g, co in cos.items():
        _compare_chunk(opt, co, g, f"chunk {g}")
    opt.materialize_errors()
    torch.cuda.synchronize()
    for g, co in cos.items():
        _compare_chunk_errors_and_p(opt, co, f"chunk {g}")
    opt.close()


def test_gpt_1p3b_bf16_5_warmup_10_compressed():
    """1,315,723,264 parameters (292 tensors), W = 4, bf16 gradients, chunk
    2^20: 5 warmup steps then 10 compressed steps, the configuration's
    counts, in the launch configuration bench.py times."""
    _run_adam_from_warmup(synth.workload("gpt-1.3b"), 5, 10, need_bytes=80e9)


def test_bert_base_100_warmup_50_compressed():
    """109,482,240 parameters (199 tensors), W = 8, fp32, chunk 2^20: the
    configuration's 100 warmup and 50 compressed steps."""
    _run_adam_from_warmup(synth.workload("bert-base"), 100, 50, need_bytes=30e9)


@pytest.mark.parametrize("n,W,chunk", [
    (1 << 30, 16, 1 << 20),   # the sweep's largest point
    (1 << 30, 1, 1 << 20),
    (1 << 26, 2, 1 << 12),    # the smallest chunk
    ((1 << 24) + 12345, 5, 1 << 16),
])
def test_sweep_points(n, W, chunk):
    wl = synth.workload("flat", n=n, W=W, chunk=chunk)
    need = n * (8 * W + 32) * 1.05
    _run_adam_fullsize(wl, steps=2, need_bytes=need)


def test_int8_full_size_sampled():
    """The INT8 quantizer at n = 2^30 + 100 (a short last block): sampled
    blocks against the oracle; the code range and the block scales'
    relation to the block maxima everywhere."""
    n = (1 << 30) + 100
    if _free_bytes() < 20e9:
        pytest.skip("needs 20 GB")
    g = torch.randn(n, generator=_gen(5), device="cuda") * 1e-3
    q = torch.empty(n, dtype=torch.int8, device="cuda")
    nb = (n + 255) // 256
    sc = torch.empty(nb, device="cuda")
    ob.ob_quant_int8(g, q, sc, 1234, 3)
    torch.cuda.synchronize()
    assert int(q.min()) >= -127 and int(q.max()) <= 127
    bmax = torch.nn.functional.pad(g.abs(), (0, nb * 256 - n)).view(-1, 256).amax(dim=1)
    # scale = max/127 rounded once: 127*scale is within one unit of max
    err = (sc.double() * 127 - bmax.double()).abs()
    assert bool((err <= torch.finfo(torch.float32).eps * bmax.double()).all())
    for b0 in (0, 1, nb // 2, nb - 2, nb - 1):
        k0 = b0 * 256
        k1 = min(n, k0 + 256)
        qo, so = O.quant_int8(host(g[k0:k1]).copy(), 256, 1234, 3, k0=k0)
        assert np.array_equal(host(q[k0:k1]), qo), f"block {b0}"
        assert_bits_equal(host(sc[b0:b0 + 1]), so, f"scale of block {b0}")


# ---------------------------------------------------------------------------
# 1-bit LAMB on the BERT-large list
# ---------------------------------------------------------------------------

def _fill_lamb_state(opt, wl, seed):
    """_fill_state plus per-layer LAMB state: sigma_l = 10^U(-1,1),
    c_avg = 10^U(-0.5,0.5), r_prev = 1, c_prev = c_prev2 = c_avg."""
    _fill_state(opt, wl, seed)
    L = wl.n_layers
    rng = np.random.default_rng(seed)
    ls0 = {"s": (10.0 ** rng.uniform(-1, 1, L)).astype(f32),
           "c_avg": (10.0 ** rng.uniform(-0.5, 0.5, L)).astype(f32)}
    ls0["r_prev"] = np.ones(L, f32)
    ls0["c_prev"] = ls0["c_avg"].copy()
    ls0["c_prev2"] = ls0["c_avg"].copy()
    for k, v in ls0.items():
        getattr(opt.ls, k).copy_(torch.from_numpy(v))
    return ls0


def _layer_slices(off, s, r):
    """Layers intersecting [s, s+r), as local offsets and global ids."""
    l0 = int(np.searchsorted(off, s, side="right") - 1)
    l1 = int(np.searchsorted(off, s + r - 1, side="right") - 1)
    ids = list(range(l0, l1 + 1))
    loc = [0] + [int(min(off[l + 1], s + r) - s) for l in ids]
    return ids, np.array(loc, np.uint64)


def test_bert_large_lamb_full_size():
    """336,226,108 parameters (302 tensors), W = 8, 1-bit LAMB, one
    compressed step from a directly drawn state (c_prev = c_prev2 = c_avg,
    so the error-feedback ratio is 1).  Exact: compression, server, pass A
    on the sampled chunks; c_t and p for every layer that lies inside a
    sampled chunk.  For all other layers: the clip bounds of r_t and c_t,
    and p moved by one common factor lr*c_t per layer."""
    wl = synth.workload("bert-large")
    if _free_bytes() < 40e9:
        pytest.skip("needs 40 GB")
    off = wl.layer_offsets.astype(np.int64)
    opt = ob.OneBitOptimizer(wl.n, wl.W, wl.chunk, wl.align, wl.grad_dtype,
                             [int(x) for x in off], lamb=True, **wl.hp)
    L = wl.n_layers
    hp = wl.hp
    std = _std_vector(wl, opt.n_pad)
    ls0 = _fill_lamb_state(opt, wl, seed=7)
    lay = opt.layout
    P, C, cpp = lay["P"], lay["chunk"], lay["chunks_per_partition"]
    chunks = _chunks(lay, wl.n)
    # also the chunk holding the embedding LayerNorm (small whole layers)
    k = int(off[3])
    j, kc = divmod(k, P)[0], (k - divmod(k, P)[0] * P) // C
    g_ln = j * cpp + kc
    if all(c[0] != g_ln for c in chunks):
        s = j * P + kc * C
        ln = min(C, P - kc * C)
        chunks.append((g_ln, s, ln, min(ln, wl.n - s)))
    st0 = _slices(opt, chunks)
    cos = {}
    for g, s, ln, r in chunks:
        ids, loc = _layer_slices(off, s, r)
        co = ChunkOracle(wl.W, s, ln, r, st0[g], O.Layers(loc))
        co.ids = ids
        co.ls = {k: v[ids].copy() for k, v in ls0.items()}
        co.full = [i for i, l in enumerate(ids) if off[l] >= s and off[l + 1] <= s + r]
        cos[g] = co
    assert any(co.full for co in cos.values()), "no whole layer inside the sampled chunks"
    p_before = {g: host(opt.p[s:s + r]).copy() for g, s, ln, r in chunks}

    grads = _grads(opt, wl, 100, std)
    gsl = _grad_slices(grads, chunks)
    opt.compressed_step(grads)
    torch.cuda.synchronize()
    assert ob.ob_device_error(opt.ctx) == 0
    c_gpu = host(opt.ls.c_t).copy()
    r_gpu = host(opt.ls.r_prev).copy()
    # clip bounds ([LAMB] paragraph 1 and 3) for every layer
    lo = np.maximum((1 - f32(hp["r_thr"])) * ls0["r_prev"], hp["r_min"])
    hi = np.minimum((1 + f32(hp["r_thr"])) * ls0["r_prev"], hp["r_max"])
    assert np.all(r_gpu >= lo * (1 - 1e-6)) and np.all(r_gpu <= hi * (1 + 1e-6))
    assert np.all(c_gpu >= hp["c_min"] * (1 - 1e-6)) and np.all(c_gpu <= hp["c_max"] * (1 + 1e-6))
    assert np.array_equal(host(opt.ls.c_prev2), ls0["c_prev"])
    for g, co in cos.items():
        S = co.state
        sigma = co.ls["s"]
        for w in range(wl.W):
            b, sc, _ = O.compress_worker(co.lay, co.grads(gsl[g])[w], S.m, S.e[w], hp["b1"],
                                         S.layers, sigma, None)
            S.bits[w], S.scales[w] = b, sc
        S.sbits, S.sscales, _ = O.server_reduce(co.lay, S.bits, S.scales, S.e_s, S.layers, None)
        R = O.lamb_pass_a(co.lay, S.layers, sigma, S.sbits, S.sscales, S.v, hp["b1"], hp["b2"],
                          S.m, S.v_fresh)
        _compare_chunk(opt, co, g, f"chunk {g}")
        if co.full:
            sub = {k: v[co.full].copy() for k, v in co.ls.items()}
            c_full = O.lamb_ratio(R[co.full], hp, sub)
            for j2, i in enumerate(co.full):
                assert_bits_equal(c_gpu[co.ids[i]], c_full[j2], f"c of layer {co.ids[i]}")
                assert_bits_equal(r_gpu[co.ids[i]], sub["r_prev"][j2], f"r of layer {co.ids[i]}")
            c_loc = np.zeros(len(co.ids), f32)
            c_loc[co.full] = c_full
            p_o = S.p.copy()
            O.lamb_pass_b(co.lay, S.layers, c_loc, S.m, S.v, hp["eps"], hp["lr"], p_o)
            loc = S.layers.off.astype(np.int64)
            p_g = host(opt.p[co.s:co.s + co.r])
            for i in co.full:
                a, b2 = loc[i], loc[i + 1]
                assert_bits_equal(p_g[a:b2], p_o[a:b2], f"p of layer {co.ids[i]}")
        # every layer in the chunk moved p by one factor lr*c_t
        loc = S.layers.off.astype(np.int64)
        u = S.m[: co.r].astype(np.float64) / (np.sqrt(S.v[: co.r].astype(np.float64)) + hp["eps"])
        dp = p_before[g].astype(np.float64) - host(opt.p[co.s:co.s + co.r]).astype(np.float64)
        for i, l in enumerate(co.ids):
            a, b2 = loc[i], loc[i + 1]
            big = np.abs(u[a:b2]) > 1e-3 * np.abs(u[a:b2]).max()
            implied = dp[a:b2][big] / u[a:b2][big] / hp["lr"]
            assert np.allclose(implied, c_gpu[l], rtol=1e-3), f"layer {l}"
    opt.materialize_errors()
    torch.cuda.synchronize()
    for g, co in cos.items():
        _compare_chunk_errors_and_p(opt, co, f"chunk {g}", p_exact=False)
    opt.close()


def test_bert_large_lamb_sign_form_equals_dense_full_size():
    """The property the sign-form momentum rests on, at full size: 1-bit
    LAMB on the BERT-large list for 4 compressed steps with the momentum
    held as the server's sign words (double-buffered, from the second step
    on) gives bit for bit the results of the dense momentum -- parameters,
    server words and scales, fresh variance, every layer's r and c, and m
    itself (rebuilt from the signs).  The dense path is the one checked
    against the oracle on sampled chunks above."""
    wl = synth.workload("bert-large")
    if _free_bytes() < 80e9:
        pytest.skip("needs 80 GB")
    off = [int(x) for x in wl.layer_offsets]
    out = []
    for sm in (False, True):
        opt = ob.OneBitOptimizer(wl.n, wl.W, wl.chunk, wl.align, wl.grad_dtype, off, lamb=True,
                                 sign_momentum=sm, **wl.hp)
        std = _std_vector(wl, opt.n_pad)
        _fill_lamb_state(opt, wl, seed=11)
        for t in range(4):
            grads = _grads(opt, wl, 300 + t, std)
            opt.compressed_step(grads)
            del grads
        torch.cuda.synchronize()
        assert ob.ob_device_error(opt.ctx) == 0
        assert opt.m_in_signs == sm
        opt.materialize_m()
        torch.cuda.synchronize()
        out.append({"p": host(opt.p), "m": host(opt.m), "v_fresh": host(opt.v_fresh),
                    "sbits": host(opt.sbits), "sscales": host(opt.sscales),
                    "e_s": host(opt.err_s), "e0": host(opt.err[0]),
                    "c_t": host(opt.ls.c_t), "r_prev": host(opt.ls.r_prev),
                    "c_prev2": host(opt.ls.c_prev2)})
        del std
        opt.close()
        torch.cuda.empty_cache()
    for k in out[0]:
        assert_bits_equal(out[1][k], out[0][k], f"{k}: sign form vs dense")


def _host_avail_bytes():
    try:
        return os.sysconf("SC_AVPHYS_PAGES") * os.sysconf("SC_PAGE_SIZE")
    except (ValueError, OSError, AttributeError):
        return 0


def test_bert_large_lamb_whole_buffer_3_warmup_10_compressed():
    """1-bit LAMB on the whole BERT-large list (336,226,108 parameters, 302
    tensors, W = 8, fp32): 3 warmup steps, the end of warmup, then 10
    compressed steps with the gradient std falling 10x over them (v_t falls
    100x, so r_t moves and its clip acts; rho = c_{t-2}/c_{t-1} differs
    from 1 from the third compressed step on).  The oracle runs the whole
    buffer -- every layer whole, so every layer's R, r and c is the
    oracle's own -- with the compressed step split over the partitions on a
    thread pool (tests/oracle_parallel.py, bit for bit the whole-buffer
    step).  The GPU runs it twice, with the dense momentum and with the
    momentum in sign form (server output double-buffered, as bench.py
    runs it), and both are compared with the oracle after every step (c
    of every layer, server words and scales) and, at the end, on every
    element of every buffer."""
    wl = synth.workload("bert-large")
    if _free_bytes() < 60e9:
        pytest.skip("needs 60 GB of free device memory")
    if _host_avail_bytes() < 48e9:
        pytest.skip("needs 48 GB of free host memory for the whole-buffer oracle")
    hp = wl.hp
    off = wl.layer_offsets.astype(np.uint64)
    opts = {sm: ob.OneBitOptimizer(wl.n, wl.W, wl.chunk, wl.align, wl.grad_dtype,
                                   [int(x) for x in off], lamb=True, sign_momentum=sm, **hp)
            for sm in (False, True)}
    n, n_pad = wl.n, opts[False].n_pad
    lay = O.Layout(n, wl.W, wl.align, wl.chunk)
    assert lay.n_pad == n_pad
    layers = O.Layers(off)
    st = O.State(lay, layers, lamb=True)
    std = _std_vector(wl, n_pad)
    p0 = torch.zeros(n_pad, device="cuda")
    p0[:n] = torch.randn(n, generator=_gen(synth.SEED_BASE + 17), device="cuda") * 0.02
    for o in opts.values():
        o.p.copy_(p0)
    st.p[:] = host(p0)
    del p0
    warm, steps = 3, 10
    with ThreadPoolExecutor(os.cpu_count() or 8) as pool:
        for t in range(warm):
            grads = _grads(opts[False], wl, t, std)
            for o in opts.values():
                o.warmup_step(grads)
            gh = [host(x) for x in grads]
            del grads
            c = O.warmup_step(lay, gh, 1, hp, st.m, st.v, st.p, layers, st.c_sum)
            torch.cuda.synchronize()
            for sm, o in opts.items():
                assert_bits_equal(host(o.ls.c_t), c, f"warmup c at step {t} (sign form {sm})")
            del gh
        for o in opts.values():
            o.begin_compression()
        O.begin_compression(st, warm, lamb=True)
        torch.cuda.synchronize()
        for sm, o in opts.items():
            for k in ("s", "c_avg", "r_prev", "c_prev", "c_prev2"):
                assert_bits_equal(host(getattr(o.ls, k)), st.ls[k], f"begin: {k} (sign form {sm})")
        for t in range(warm, warm + steps):
            f = 10.0 ** (-(t - warm) / (steps - 1))
            grads = _grads(opts[False], wl, t, std * f)
            for o in opts.values():
                o.compressed_step(grads)
            gh = [host(x) for x in grads]
            del grads
            OP.compressed_step(st, gh, hp, pool, lamb=True)
            del gh
            torch.cuda.synchronize()
            for sm, o in opts.items():
                what = f"step {t} (sign form {sm})"
                assert_bits_equal(host(o.ls.c_t), st.c, f"c of every layer, {what}")
                assert_bits_equal(host(o.sscales), st.sscales, f"server scales, {what}")
                assert_bits_equal(host(o.sbits)[: lay.words], st.sbits, f"server words, {what}")
    assert np.any(st.ls["r_prev"] != 1.0), "the ratio never moved"
    assert np.any(st.ls["c_prev"] != st.ls["c_prev2"]), "rho stayed 1"
    for sm, o in opts.items():
        assert ob.ob_device_error(o.ctx) == 0
        what = f"(sign form {sm})"
        for k in ("r_prev", "c_prev", "c_prev2"):
            assert_bits_equal(host(getattr(o.ls, k)), st.ls[k], f"{k} {what}")
        o.materialize_m()
        assert_bits_equal(host(o.bits)[:, : lay.words], st.bits, f"worker words {what}")
        assert_bits_equal(host(o.scales), st.scales, f"worker scales {what}")
        o.materialize_errors()
        torch.cuda.synchronize()
        pairs = [("m", o.m, st.m), ("p", o.p, st.p), ("e_s", o.err_s, st.e_s),
                 ("v_fresh", o.v_fresh, st.v_fresh)]
        pairs += [(f"e[{w}]", o.err[w], st.e[w]) for w in range(wl.W)]
        for name, gbuf, want in pairs:
            got = host(gbuf)
            assert_close(got, want, f"{name} {what}")
            assert_bits_equal(got, want, f"{name} {what}")
        o.close()
    torch.cuda.empty_cache()
