"""Parity of the CUDA path (through the C ABI) with the oracle, element by
element, on the same seeded inputs.

Bar: packed sign words, INT8 codes and scales bit-exact; every float buffer
bit-exact as well for single kernels (both sides round every operation the
same way and sum in the same fixed order), and within rel 1e-5 / abs 1e-7
after multi-step runs.
"""
import numpy as np
import pytest
import torch

import momentum_compression_gb300 as ob
import oracle as O
import synth
from helpers import (Guarded, assert_bits_equal, assert_close, assert_guards, bf16_tensor, dev,
                     host)

pytestmark = pytest.mark.gpu

f32 = np.float32


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)
    from momentum_compression_gb300 import _build
    _build.build()
    yield
    torch.cuda.synchronize()


# (n, W, align, chunk, grad dtype)
CASES = [
    (1 << 20, 4, 4096, 1 << 18, "f32"),      # the flat 2^20 workload
    (50_037, 3, 32, 992, "f32"),             # chunk not a multiple of the tile
    (4097, 2, 32, 64, "bf16"),
    (1, 1, 32, 32, "f32"),
    (31, 2, 32, 32, "f32"),
    (33, 3, 32, 64, "f32"),
    (4095, 1, 4096, 4096, "f32"),
    (100, 4, 4096, 1 << 20, "f32"),          # partitions 1..3 are all padding
    (70_001, 16, 4096, 4096, "bf16"),
    (9_000, 64, 32, 32, "f32"),              # the largest W
    (300_000, 5, 4096, 3 * 4096 + 32, "f32"),  # ragged last tile of each chunk
]


def _ids(c):
    return "n{}-W{}-A{}-C{}-{}".format(*c)


class Case:
    def __init__(self, n, W, A, C, dt, seed=0):
        self.n, self.W, self.A, self.C, self.dt = n, W, A, C, dt
        self.lay = O.Layout(n, W, A, C)
        self.ctx = ob.ob_init(n, W, C, A, ob.OB_GRAD_BF16 if dt == "bf16" else ob.OB_GRAD_F32,
                              b1=0.9, b2=0.999, eps=1e-8, lr=1e-4)
        lay = ob.ob_get_layout(self.ctx)
        assert (lay["n_pad"], lay["P"], lay["n_chunks"]) == (self.lay.n_pad, self.lay.P,
                                                            self.lay.nc)
        self.words = lay["words_per_worker"]  # row stride, >= the oracle's word count
        assert self.words >= self.lay.words and self.words % 4 == 0
        nb = ob.ob_workspace_bytes(self.ctx)
        self.ws = torch.zeros((nb + 255) // 4, dtype=torch.float32, device="cuda")
        ob.ob_set_workspace(self.ctx, self.ws, nb)
        self.rng = np.random.default_rng(seed + n + 7 * W)

    def vec(self, scale, fill=0.0):
        a = np.full(self.lay.n_pad, fill, f32)
        a[: self.n] = self.rng.standard_normal(self.n).astype(f32) * f32(scale)
        return a

    def grads(self, scale=1e-3):
        g = [self.vec(scale) for _ in range(self.W)]
        if self.dt == "bf16":
            bits = [synth.bf16_bits(x) for x in g]
            return [synth.bf16_to_f32(b) for b in bits], [bf16_tensor(b) for b in bits]
        return g, [dev(x) for x in g]

    def close(self):
        ob.ob_destroy(self.ctx)


def _materialize(c, err_t, bits_t, scales_t, es_t, sbits_t, sscales_t):
    ob.ob_materialize_errors(c.ctx, err_t, bits_t, scales_t, es_t, sbits_t, sscales_t)


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_compress_server_update_single_kernels(case):
    """Each kernel of the step on the same inputs as the oracle, bit for
    bit, with every buffer a call writes (and m, which it must not) in a
    guarded allocation whose poisoned margins are checked after each call;
    then the error monitor on the same deferred state."""
    c = Case(*case)
    lay = c.lay
    g_host, g_dev = c.grads()
    m = c.vec(1e-3)
    e = [c.vec(1e-4) for _ in range(c.W)]
    # --- worker compression
    err_g = [Guarded(lay.n_pad, torch.float32, x) for x in e]  # deferred form, zero scales
    err_t = [x.t for x in err_g]
    bits_g = Guarded((c.W, c.words), torch.int32, np.zeros((c.W, c.words), np.int32))
    scales_g = Guarded((c.W, lay.nc), torch.float32, np.zeros((c.W, lay.nc), f32))
    m_g = Guarded(lay.n_pad, torch.float32, m)
    bits_t, scales_t, m_t = bits_g.t, scales_g.t, m_g.t
    ob.ob_compress(c.ctx, g_dev, m_t, err_t, bits_t, scales_t)
    torch.cuda.synchronize()
    assert_guards("compress", bits_g, scales_g, m_g, *err_g)
    bits_o = np.zeros((c.W, lay.words), np.uint32)
    scales_o = np.zeros((c.W, lay.nc), f32)
    e_o = [x.copy() for x in e]
    for w in range(c.W):
        b, s, x = O.compress_worker(lay, g_host[w], m, e_o[w], 0.9)
        bits_o[w], scales_o[w] = b, s
        assert_bits_equal(host(err_t[w]), x, f"x of worker {w}")
    assert_bits_equal(host(bits_t)[:, : lay.words], bits_o, "worker sign words")
    assert not host(bits_t)[:, lay.words:].any()
    assert_bits_equal(host(scales_t), scales_o, "worker scales")
    assert_bits_equal(host(m_t), m, "m is read only")
    # --- server
    es = c.vec(1e-4)
    es_g = Guarded(lay.n_pad, torch.float32, es)
    sbits_g = Guarded(c.words, torch.int32, np.zeros(c.words, np.int32))
    sscales_g = Guarded(lay.nc, torch.float32, np.zeros(lay.nc, f32))
    es_t, sbits_t, sscales_t = es_g.t, sbits_g.t, sscales_g.t
    ob.ob_server_reduce(c.ctx, bits_t, scales_t, es_t, sbits_t, sscales_t)
    torch.cuda.synchronize()
    assert_guards("server", es_g, sbits_g, sscales_g, bits_g, scales_g)
    es_o = es.copy()
    sbits_o, sscales_o, y_o = O.server_reduce(lay, bits_o, scales_o, es_o)
    assert ob.ob_device_error(c.ctx) == 0
    assert_bits_equal(host(es_t), y_o, "server y")
    assert_bits_equal(host(sbits_t)[: lay.words], sbits_o, "server sign words")
    assert_bits_equal(host(sscales_t), sscales_o, "server scales")
    # --- the error monitor on the deferred state: per chunk, the sums of
    # the squared true errors of every worker and of the server
    norm_g = Guarded((c.W + 1, lay.nc), torch.float32, np.full((c.W + 1, lay.nc), 5.0, f32))
    ob.ob_error_norm(c.ctx, err_t, bits_t, scales_t, es_t, sbits_t, sscales_t, norm_g.t)
    torch.cuda.synchronize()
    assert_guards("error_norm", norm_g)
    got = host(norm_g.t)
    for w in range(c.W):
        assert_bits_equal(got[w], O.error_norm(lay, e_o[w]), f"error norm of worker {w}")
    assert_bits_equal(got[c.W], O.error_norm(lay, es_o), "error norm of the server")
    # --- decompression and the Adam update
    out_g = Guarded(lay.n_pad, torch.float32, np.full(lay.n_pad, 7.0, f32))
    ob.ob_decompress(c.ctx, sbits_t, sscales_t, out_g.t)
    torch.cuda.synchronize()
    assert_guards("decompress", out_g)
    assert_bits_equal(host(out_g.t), O.decompress(lay, sbits_o, sscales_o), "decompress")
    v = np.abs(c.vec(1e-6)) + f32(1e-12)
    p = c.vec(0.02)
    v_t = dev(v)
    p_g = Guarded(lay.n_pad, torch.float32, p)
    m2_g = Guarded(lay.n_pad, torch.float32, np.full(lay.n_pad, 3.0, f32))
    ob.ob_adam_step(c.ctx, sbits_t, sscales_t, v_t, m2_g.t, p_g.t)
    torch.cuda.synchronize()
    assert_guards("adam_step", p_g, m2_g)
    m_o = np.full(lay.n_pad, 3.0, f32)
    p_o = p.copy()
    O.adam_update(lay, sbits_o, sscales_o, v, 1e-8, 1e-4, m_o, p_o)
    assert_bits_equal(host(m2_g.t), m_o, "m after update")
    assert_bits_equal(host(p_g.t), p_o, "p after update")
    # --- deferred errors made explicit
    _materialize(c, err_t, bits_t, scales_t, es_t, sbits_t, sscales_t)
    torch.cuda.synchronize()
    assert_guards("materialize", es_g, scales_g, sscales_g, *err_g)
    for w in range(c.W):
        assert_bits_equal(host(err_t[w]), e_o[w], f"e' of worker {w}")
    assert_bits_equal(host(es_t), es_o, "server e'")
    assert not host(scales_t).any() and not host(sscales_t).any()
    c.close()


def _run_adam(wl, warm, steps, check_every=False, sign_momentum=False, reset_interval=0,
              clip=0.0):
    """Runs `warm` warmup and `steps` compressed steps of workload wl on the
    GPU and in the oracle from the same seeded inputs."""
    n, W = wl.n, wl.W
    opt = ob.OneBitOptimizer(n, W, wl.chunk, wl.align, wl.grad_dtype,
                             sign_momentum=sign_momentum, reset_interval=reset_interval,
                             clip_value=clip, **wl.hp)
    hp_o = dict(wl.hp, clip=clip)
    lay = O.Layout(n, W, wl.align, wl.chunk)
    st = O.State(lay)
    p0 = np.zeros(lay.n_pad, f32)
    p0[:n] = synth.params0_slice(wl, 0, n)
    st.p[:] = p0
    opt.p.copy_(torch.from_numpy(p0))

    def grads(step):
        gh = []
        gd = []
        for w in range(W):
            a = np.zeros(lay.n_pad, f32)
            a[:n] = synth.grad_slice(wl, step, w, 0, n)
            if wl.grad_dtype == "bf16":
                b = synth.bf16_bits(a)
                gh.append(synth.bf16_to_f32(b))
                gd.append(bf16_tensor(b))
            else:
                gh.append(a)
                gd.append(dev(a))
        return gh, gd

    for t in range(warm):
        gh, gd = grads(t)
        opt.warmup_step(gd)
        O.warmup_step(lay, gh, 0, wl.hp, st.m, st.v, st.p)
    torch.cuda.synchronize()
    assert_bits_equal(host(opt.m), st.m, "m after warmup")
    assert_bits_equal(host(opt.v), st.v, "v after warmup")
    assert_bits_equal(host(opt.p), st.p, "p after warmup")
    opt.begin_compression()
    O.begin_compression(st, warm)
    for t in range(warm, warm + steps):
        gh, gd = grads(t)
        opt.compressed_step(gd)
        c = t - warm
        if reset_interval and c and c % reset_interval == 0:
            O.reset_errors(st)
        O.compressed_step(st, gh, hp_o)
        if check_every:
            torch.cuda.synchronize()
            assert_bits_equal(host(opt.sbits)[: lay.words], st.sbits, f"sbits at step {t}")
    torch.cuda.synchronize()
    return opt, st, lay


def _compare_state(opt, st, lay, exact=True):
    assert ob.ob_device_error(opt.ctx) == 0
    norms = host(opt.error_norm())  # from the deferred state, before it is made explicit
    for w in range(lay.W):
        assert_bits_equal(norms[w], O.error_norm(lay, st.e[w]), f"error norm of worker {w}")
    assert_bits_equal(norms[lay.W], O.error_norm(lay, st.e_s), "error norm of the server")
    opt.materialize_m()
    assert_bits_equal(host(opt.sbits)[: lay.words], st.sbits, "server sign words")
    assert_bits_equal(host(opt.sscales), st.sscales, "server scales")
    assert_bits_equal(host(opt.bits)[:, : lay.words], st.bits, "worker sign words")
    assert_bits_equal(host(opt.scales), st.scales, "worker scales")
    opt.materialize_errors()
    torch.cuda.synchronize()
    pairs = [("m", opt.m, st.m), ("p", opt.p, st.p), ("e_s", opt.err_s, st.e_s)]
    pairs += [(f"e[{w}]", opt.err[w], st.e[w]) for w in range(lay.W)]
    if opt.v_fresh is not None:
        pairs.append(("v_fresh", opt.v_fresh, st.v_fresh))
    for name, g, o in pairs:
        assert_close(host(g), o, name)
        if exact:
            assert_bits_equal(host(g), o, name)


def test_flat_1m_adam_5_warmup_10_compressed():
    """The flat 2^20-element workload: W = 4, chunk 2^18, 5 uncompressed
    warmup steps then 10 compressed steps."""
    wl = synth.workload("flat-1m")
    opt, st, lay = _run_adam(wl, wl.warmup_steps, wl.compressed_steps, check_every=True)
    _compare_state(opt, st, lay)
    opt.close()


@pytest.mark.parametrize("workload,dt,W", [
    ("flat-1m", "f32", None), ("gpt-1.3b", "bf16", None),
    # the worker kernel takes workers in groups of 4 in sign form: a ragged
    # last group (5 = 4 + 1), four full groups (16), and bf16 with 6
    ("flat", "f32", 5), ("flat", "f32", 16), ("flat", "bf16", 6),
    ("flat", "f32", 64),  # the largest W: 16 groups, the generic server
])
def test_sign_momentum_matches_oracle(workload, dt, W):
    """1-bit Adam with the momentum held as the server's sign words and
    chunk scales (ob_compress_signm, ob_adam_step without m): the same
    results as the dense momentum, bit for bit; the dense m, rebuilt by
    ob_decompress, equals the oracle's."""
    if workload == "flat":
        wl = synth.workload("flat", n=150_001 if W < 64 else 40_003, W=W, chunk=1 << 13,
                            grad_dtype=dt)
    else:
        wl = synth.workload(workload)
    if workload == "gpt-1.3b":
        wl.tensors = None
        wl.n = 250_000
        wl.chunk = 1 << 13
    opt, st, lay = _run_adam(wl, 2, 6, check_every=True, sign_momentum=True)
    assert opt.m_in_signs
    _compare_state(opt, st, lay)
    opt.close()


@pytest.mark.parametrize("sign_momentum", [False, True])
def test_stability_variants(sign_momentum):
    """The "1bit Adam" write-up's stability variants (4.1): the compensated
    value clamped to +-clip_value and the errors reset every 3 steps, for 8
    steps -- against the oracle, bit for bit."""
    wl = synth.workload("flat", n=200_003, W=3, chunk=1 << 14)
    opt, st, lay = _run_adam(wl, 2, 8, check_every=True, sign_momentum=sign_momentum,
                             reset_interval=3, clip=2.5e-4)
    _compare_state(opt, st, lay)
    opt.close()


def test_bf16_gpt_shaped_slice_adam():
    """bf16 gradients on the first 300,000 parameters of the GPT-1.3B list
    (wte rows), W = 4, chunk 2^14, 2 warmup + 4 compressed steps."""
    wl = synth.workload("gpt-1.3b")
    wl.tensors = None
    wl.n = 300_000
    wl.chunk = 1 << 14
    opt, st, lay = _run_adam(wl, 2, 4)
    _compare_state(opt, st, lay)
    opt.close()


def test_deferred_resume_is_bit_identical():
    """Materialising the errors between steps (as before a checkpoint) does
    not change any later result."""
    wl = synth.workload("flat", n=200_003, W=3, chunk=1 << 14)
    a, st, lay = _run_adam(wl, 2, 3)
    gd = [dev(synth.grad_slice(wl, 9, w, 0, lay.n_pad)) for w in range(3)]
    a.materialize_errors()
    a.compressed_step(gd)
    b, _, _ = _run_adam(wl, 2, 3)
    b.compressed_step(gd)
    torch.cuda.synchronize()
    for x, y in ((a.p, b.p), (a.m, b.m), (a.sbits, b.sbits)):
        assert torch.equal(x, y)
    a.materialize_errors()
    b.materialize_errors()
    torch.cuda.synchronize()
    for w in range(3):
        assert torch.equal(a.err[w], b.err[w])
    a.close()
    b.close()


# ---------------------------------------------------------------------------
# 1-bit LAMB
# ---------------------------------------------------------------------------

LAMB_HP = dict(b1=0.9, b2=0.999, eps=1e-6, lr=1e-3, r_thr=0.1, r_min=0.5, r_max=4.0,
               c_min=0.01, c_max=10.0)


@pytest.mark.parametrize("flags,W,dt,sm,warm,steps", [
    (0, 4, "f32", False, 3, 6), (ob.OB_FLAG_NO_RATIO_EF, 4, "f32", False, 3, 6),
    (ob.OB_FLAG_FROZEN_C, 4, "f32", False, 3, 6),
    (0, 8, "bf16", False, 3, 6),   # the W = 8 server specialisation, bf16 worker kernel
    (0, 3, "f32", False, 3, 6),    # generic W
    (0, 12, "bf16", False, 3, 6),  # workers beyond the 8-worker sign table
    # the momentum in sign form, server output double-buffered
    (0, 4, "f32", True, 3, 6), (ob.OB_FLAG_NO_RATIO_EF, 3, "f32", True, 3, 6),
    (ob.OB_FLAG_FROZEN_C, 8, "bf16", True, 3, 6), (0, 12, "bf16", True, 3, 6),
    (ob.OB_FLAG_NO_RATIO_EF, 16, "f32", True, 3, 6),  # the W = 16 server specialisation
    (0, 64, "f32", True, 3, 6),                       # the largest W, the generic server
    # the BERT-large LAMB configuration's step counts (W = 8, fp32, 10
    # warmup + 50 compressed steps, v falling 100x over the compressed
    # steps) under each flag setting, sign form and dense
    (0, 8, "f32", True, 10, 50), (ob.OB_FLAG_NO_RATIO_EF, 8, "f32", True, 10, 50),
    (ob.OB_FLAG_FROZEN_C, 8, "f32", True, 10, 50), (0, 8, "f32", False, 10, 50),
])
def test_lamb_small_layers(flags, W, dt, sm, warm, steps):
    """Layers of odd sizes (1, 2, 7, 4095, 4097, ...) fused into one buffer,
    chunk 2048, `warm` warmup + `steps` compressed steps with the gradient
    std falling over the compressed steps (3x per step in the short runs,
    10x over the 50 steps of the long ones), so that r_t moves and the
    step-ratio error feedback differs from 1.  sm: the momentum held as
    sscale*sign/sigma_l of the server output (ob_step_db from the second
    compressed step on), which must give the dense path's results bit for
    bit."""
    sizes = [7, 1, 2, 4095, 4097, 33, 1000, 20000, 3, 30000]
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.uint64)
    n, A, C = int(off[-1]), 32, 2048
    opt = ob.OneBitOptimizer(n, W, C, A, dt, [int(x) for x in off], lamb=True, flags=flags,
                             sign_momentum=sm, **LAMB_HP)
    lay = O.Layout(n, W, A, C)
    layers = O.Layers(off)
    st = O.State(lay, layers, lamb=True)
    rng = np.random.default_rng(3)
    p0 = np.zeros(lay.n_pad, f32)
    p0[:n] = rng.standard_normal(n).astype(f32) * f32(0.02)
    st.p[:] = p0
    opt.p.copy_(torch.from_numpy(p0))
    layer_std = np.repeat(10.0 ** rng.uniform(-4, -2, size=len(sizes)), sizes).astype(f32)

    def decay(t):
        k = max(0, t - warm)
        return f32(3.0 ** -k) if steps <= 6 else f32(10.0 ** (-k / (steps - 1)))

    def grads(t):
        f = decay(t)
        gh = []
        for w in range(W):
            a = np.zeros(lay.n_pad, f32)
            a[:n] = rng.standard_normal(n).astype(f32) * layer_std * f
            gh.append(a)
        if dt == "bf16":
            bits = [synth.bf16_bits(x) for x in gh]
            return [synth.bf16_to_f32(b) for b in bits], [bf16_tensor(b) for b in bits]
        return gh, [dev(x) for x in gh]

    hp = dict(LAMB_HP)
    for t in range(warm):
        gh, gd = grads(t)
        opt.warmup_step(gd)
        c = O.warmup_step(lay, gh, 1, hp, st.m, st.v, st.p, layers, st.c_sum)
        torch.cuda.synchronize()
        assert_bits_equal(host(opt.ls.c_t), c, f"warmup c at step {t}")
    assert_bits_equal(host(opt.m), st.m, "m after warmup")
    assert_bits_equal(host(opt.v), st.v, "v after warmup")
    assert_bits_equal(host(opt.p), st.p, "p after warmup")
    assert_bits_equal(host(opt.ls.c_sum), st.c_sum, "c_sum after warmup")
    opt.begin_compression()
    O.begin_compression(st, warm, lamb=True)
    torch.cuda.synchronize()
    for k in ("s", "c_avg", "r_prev", "c_prev", "c_prev2"):
        assert_bits_equal(host(getattr(opt.ls, k)), st.ls[k], f"begin: {k}")
    ratio_ef = not (flags & ob.OB_FLAG_NO_RATIO_EF)
    frozen = bool(flags & ob.OB_FLAG_FROZEN_C)
    for t in range(warm, warm + steps):
        gh, gd = grads(t)
        prev = (st.sbits.copy(), st.sscales.copy())
        opt.compressed_step(gd)
        O.compressed_step(st, gh, hp, lamb=True, ratio_ef=ratio_ef, frozen=frozen)
        torch.cuda.synchronize()
        assert_bits_equal(host(opt.sbits)[: lay.words], st.sbits, f"sbits at step {t}")
        assert_bits_equal(host(opt.sscales), st.sscales, f"sscales at step {t}")
        assert_bits_equal(host(opt.ls.c_t), st.c, f"c_t at step {t}")
        if sm and t > warm:  # the previous output is left intact in the other buffer
            assert opt.m_in_signs
            assert_bits_equal(host(opt.sbits_alt)[: lay.words], prev[0], f"old sbits at {t}")
            assert_bits_equal(host(opt.sscales_alt), prev[1], f"old sscales at {t}")
    for k in ("r_prev", "c_prev", "c_prev2"):
        assert_bits_equal(host(getattr(opt.ls, k)), st.ls[k], f"end: {k}")
    if not frozen:
        assert np.any(st.ls["r_prev"] != 1.0)
    _compare_state(opt, st, lay)
    opt.close()


# ---------------------------------------------------------------------------
# INT8
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("n", [1, 3, 4, 5, 255, 256, 257, 1000, 4097, (1 << 20) + 3])
def test_int8_parity(n):
    rng = np.random.default_rng(n)
    g = (rng.standard_normal(n) * 1e-3).astype(f32)
    if n > 600:
        g[256:512] = 0.0  # an all-zero block
        g[700] = np.float32(5.0)  # a block dominated by one value
    nb = (n + 255) // 256
    g_g = Guarded(n, torch.float32, g)
    q_g = Guarded(n, torch.int8, np.zeros(n, np.int8))
    s_g = Guarded(nb, torch.float32, np.zeros(nb, f32))
    d_g = Guarded(n, torch.float32, np.zeros(n, f32))
    for step in (0, 1, 2 ** 33 + 5):
        ob.ob_quant_int8(g_g.t, q_g.t, s_g.t, 1234, step, d_g.t, n=n)
        torch.cuda.synchronize()
        assert_guards(f"quant_int8, step {step}", g_g, q_g, s_g, d_g)
        q_o, s_o, d_o = O.quant_int8(g, 256, 1234, step, deq=True)
        assert np.array_equal(host(q_g.t), q_o), f"codes, step {step}"
        assert_bits_equal(host(s_g.t), s_o, "block scales")
        assert_bits_equal(host(d_g.t), d_o, "dequantised")


def _int8_adversarial(seed, step, nblk=96):
    """Blocks whose values put the quotient g/scale at, just above or just
    below (0 to a few times 2^-15 away) an integer plus the value's own
    uniform -- where the rounding decision flips -- and near integers, at
    +-127, inside (-1, 0); some blocks with zeros, a NaN, or a scale below
    the normal range.  The uniforms are the oracle's."""
    rng = np.random.default_rng(seed)
    n = 256 * nblk
    k = np.arange(n)
    u = np.array([O.uniform(seed, step, int(i)) for i in k], np.float64)
    deltas = np.array([0.0, 2.0 ** -24, -2.0 ** -24, 2.0 ** -20, -2.0 ** -20, 2.0 ** -17,
                       -2.0 ** -17, 5 * 2.0 ** -18, -5 * 2.0 ** -18, 2.0 ** -15, -2.0 ** -15,
                       1.5 * 2.0 ** -15, -1.5 * 2.0 ** -15, 2.0 ** -12, -2.0 ** -12])
    g = np.zeros(n, np.float32)
    for b in range(nblk):
        sl = slice(256 * b, 256 * b + 256)
        kind = b % 6
        mx = np.float32(10.0 ** rng.uniform(-6, 2)) if kind != 5 else np.float32(1e-37)
        s = np.float64(np.float32(mx / np.float32(127.0)))
        j = rng.integers(-127, 127, 256).astype(np.float64)
        if kind == 1:
            j[:] = -1.0  # quotients in (-1, 0)
        d = deltas[rng.integers(0, len(deltas), 256)]
        frac = u[sl] + d if kind != 2 else d  # kind 2: near integers
        v = np.clip(s * (j + frac), -float(mx), float(mx)).astype(np.float32)
        v[0] = mx if b % 2 else -mx
        if kind == 3:
            v[1::3] = 0.0
        if kind == 4:
            v[7] = np.nan
        g[sl] = v
    return g


@pytest.mark.parametrize("variant", ["plain", "deq", "ef"])
def test_int8_decision_adversarial(variant):
    """The codes next to every rounding decision's boundary, bit for bit with
    the oracle's (the division-free codes are taken only where provably
    equal to the division's; the rest go through the division)."""
    seed, step = 4321, 9
    g = _int8_adversarial(seed, step)
    n = g.size
    nb = n // 256
    q_g = Guarded(n, torch.int8, np.zeros(n, np.int8))
    s_g = Guarded(nb, torch.float32, np.zeros(nb, f32))
    d_g = Guarded(n, torch.float32, np.zeros(n, f32))
    if variant == "ef":
        e0 = (np.random.default_rng(2).standard_normal(n) * 1e-9).astype(f32)
        e_g = Guarded(n, torch.float32, e0)
        ob.ob_quant_int8_ef(dev(g), e_g.t, q_g.t, s_g.t, seed, step, d_g.t, None, n=n)
        q_o, s_o, d_o, _ = O.quant_int8_ef(g, e0.copy(), seed, step, deq=True, err2=True)
    else:
        ob.ob_quant_int8(dev(g), q_g.t, s_g.t, seed, step, d_g.t if variant == "deq" else None,
                         n=n)
        q_o, s_o, d_o = O.quant_int8(g, 256, seed, step, deq=True)
    torch.cuda.synchronize()
    assert_guards(f"int8 {variant}", q_g, s_g, d_g)
    assert np.array_equal(host(q_g.t), q_o), f"{(host(q_g.t) != q_o).sum()} codes differ"
    assert_bits_equal(host(s_g.t), s_o, "block scales")
    if variant != "plain":
        assert_bits_equal(host(d_g.t), d_o, "dequantised")


def test_int8_large_seed_and_no_deq():
    n = 3 * 256 + 17
    g = (np.random.default_rng(1).standard_normal(n) * 10).astype(f32)
    g_t = dev(g)
    q_t = torch.zeros(n, dtype=torch.int8, device="cuda")
    s_t = torch.zeros(4, dtype=torch.float32, device="cuda")
    seed = 0xFEDCBA9876543210
    ob.ob_quant_int8(g_t, q_t, s_t, seed, 77)
    q_o, s_o = O.quant_int8(g, 256, seed, 77)
    assert np.array_equal(host(q_t), q_o)
    assert_bits_equal(host(s_t), s_o)


# ---------------------------------------------------------------------------
# Edge cases
# ---------------------------------------------------------------------------

def test_nan_gradient_propagates_like_the_oracle():
    """A NaN gradient packs as -1 and poisons its chunk's scale, on both
    sides alike; no trap, and other chunks are untouched."""
    c = Case(40_000, 2, 32, 4096, "f32", seed=5)
    lay = c.lay
    g_host, _ = c.grads()
    g_host[1][5000] = np.nan
    g_dev = [dev(x) for x in g_host]
    m = c.vec(1e-3)
    err_t = [torch.zeros(lay.n_pad, device="cuda") for _ in range(2)]
    bits_t = torch.zeros((2, c.words), dtype=torch.int32, device="cuda")
    scales_t = torch.zeros((2, lay.nc), dtype=torch.float32, device="cuda")
    ob.ob_compress(c.ctx, g_dev, dev(m), err_t, bits_t, scales_t)
    for w in range(2):
        b, s, x = O.compress_worker(lay, g_host[w], m, np.zeros(lay.n_pad, f32), 0.9)
        assert np.array_equal(host(bits_t[w]).view(np.uint32)[: lay.words], b)
        got = host(scales_t[w])
        assert np.array_equal(np.isnan(got), np.isnan(s))
        assert_bits_equal(got[~np.isnan(s)], s[~np.isnan(s)])
    assert np.isnan(host(scales_t[1])).sum() == 1
    c.close()


def test_misaligned_pointers_rejected_before_launch():
    c = Case(4096, 2, 32, 1024, "f32")
    buf = torch.zeros(8192 + 8, device="cuda")
    bad = buf.data_ptr() + 4
    with pytest.raises(ob.OBError) as ei:
        ob.ob_adam_step(c.ctx, buf, buf, bad, buf, buf)
    assert ei.value.status == ob.OB_ERR_ALIGN
    with pytest.raises(ob.OBError) as ei:
        ob.ob_compress(c.ctx, [buf, bad], buf, [buf, buf], buf, buf)
    assert ei.value.status == ob.OB_ERR_ALIGN
    c.close()


def test_double_buffer_arguments_rejected_before_launch():
    """The double-buffered calls refuse server buffers that overlap without
    being equal, and a sign-form LAMB update whose previous and current
    buffers coincide, on the host, before any launch."""
    sizes = [1000, 3000]
    opt = ob.OneBitOptimizer(sum(sizes), 2, 2048, 32, "f32", [0, 1000, 4000], lamb=True,
                             sign_momentum=True, **LAMB_HP)
    words = opt.layout["words_per_worker"]
    big = torch.zeros(2 * words + 64, dtype=torch.int32, device="cuda")
    shifted = big[4:4 + words]  # overlaps big[:words], 16 bytes further on
    with pytest.raises(ob.OBError) as ei:
        ob.ob_server_reduce_db(opt.ctx, opt.bits, opt.scales, opt.err_s, big, opt.sscales,
                               shifted, opt.sscales_alt, opt.ls)
    assert ei.value.status == ob.OB_ERR_INVALID
    with pytest.raises(ob.OBError) as ei:
        ob.ob_lamb_step_signm(opt.ctx, opt.sbits, opt.sscales, opt.sbits, opt.sscales_alt,
                              opt.v, opt.v_fresh, opt.p, opt.ls)
    assert ei.value.status == ob.OB_ERR_INVALID
    with pytest.raises(ob.OBError) as ei:
        ob.ob_lamb_step_signm(opt.ctx, None, opt.sscales, opt.sbits_alt, opt.sscales_alt,
                              opt.v, opt.v_fresh, opt.p, opt.ls)
    assert ei.value.status == ob.OB_ERR_INVALID
    # equal pairs are the in-place server
    ob.ob_server_reduce_db(opt.ctx, opt.bits, opt.scales, opt.err_s, opt.sbits, opt.sscales,
                           opt.sbits, opt.sscales, opt.ls)
    torch.cuda.synchronize()
    assert ob.ob_device_error(opt.ctx) == 0
    opt.close()


@pytest.mark.parametrize("deq,err2", [(True, True), (False, True), (False, False)])
@pytest.mark.parametrize("n", [1, 255, 256, 1000, 4097, (1 << 20) + 5])
def test_int8_error_feedback_parity(n, deq, err2):
    """INT8 with error feedback (with and without the dequantised output and
    the per-block error monitor: each pair is its own kernel), three calls
    in a row (the residual carries over), against the oracle bit for bit."""
    rng = np.random.default_rng(n + 17)
    e_o = (rng.standard_normal(n) * 1e-5).astype(f32)
    nb = (n + 255) // 256
    e_g = Guarded(n, torch.float32, e_o)
    q_g = Guarded(n, torch.int8, np.zeros(n, np.int8))
    s_g = Guarded(nb, torch.float32, np.zeros(nb, f32))
    d_g = Guarded(n, torch.float32, np.zeros(n, f32)) if deq else None
    e2_g = Guarded(nb, torch.float32, np.zeros(nb, f32)) if err2 else None
    outs = [x for x in (d_g, e2_g) if x is not None]
    for step in range(3):
        g = (rng.standard_normal(n) * 1e-3).astype(f32)
        ob.ob_quant_int8_ef(dev(g), e_g.t, q_g.t, s_g.t, 77, step, d_g.t if deq else None,
                            e2_g.t if err2 else None, n=n)
        torch.cuda.synchronize()
        assert_guards(f"quant_int8_ef, call {step}", e_g, q_g, s_g, *outs)
        ref = O.quant_int8_ef(g, e_o, 77, step, deq=deq, err2=err2)
        q_o, s_o = ref[0], ref[1]
        assert np.array_equal(host(q_g.t), q_o), f"codes, call {step}"
        assert_bits_equal(host(s_g.t), s_o, "scales")
        if deq:
            assert_bits_equal(host(d_g.t), ref[2], "dequantised")
        assert_bits_equal(host(e_g.t), e_o, "residual")
        if err2:
            assert_bits_equal(host(e2_g.t), ref[-1], "error monitor")


# ---------------------------------------------------------------------------
# Degenerate inputs
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("lamb", [False, True])
def test_all_zero_inputs(lamb):
    """All gradients, momentum and errors zero: every chunk scale is 0,
    every sign is +1 (x = +0 >= 0), errors stay 0, and the update leaves p
    as it is -- bit for bit as the oracle.  LAMB: zero norms give c = 1."""
    n, W, A, C = 20_000, 4, 32, 4096
    off = [0, 100, 20_000] if lamb else None
    hp = dict(LAMB_HP) if lamb else dict(b1=0.9, b2=0.999, eps=1e-8, lr=1e-4)
    opt = ob.OneBitOptimizer(n, W, C, A, "f32", off, lamb=lamb, **hp)
    lay = O.Layout(n, W, A, C)
    layers = O.Layers(np.array(off, np.uint64)) if lamb else None
    st = O.State(lay, layers, lamb=lamb)
    p0 = np.zeros(lay.n_pad, f32)
    p0[:n] = np.linspace(-1, 1, n, dtype=f32)
    st.p[:] = p0
    opt.p.copy_(dev(p0))
    st.v[:n] = f32(1e-6)
    opt.v[:n] = 1e-6
    zeros = [np.zeros(lay.n_pad, f32) for _ in range(W)]
    if lamb:
        opt.warmup_step([dev(z) for z in zeros])
        O.warmup_step(lay, zeros, 1, hp, st.m, st.v, st.p, layers, st.c_sum)
    opt.begin_compression()
    O.begin_compression(st, 1, lamb=lamb)
    for t in range(2):
        opt.compressed_step([dev(z) for z in zeros])
        O.compressed_step(st, zeros, hp, lamb=lamb)
    torch.cuda.synchronize()
    assert_bits_equal(host(opt.sbits)[: lay.words], st.sbits, "sbits")
    assert np.all(st.sscales == 0) and np.all(host(opt.sscales) == 0)
    assert_bits_equal(host(opt.p), st.p, "p")
    assert_bits_equal(host(opt.p)[:n], p0[:n], "p unchanged")
    if lamb:
        assert_bits_equal(host(opt.ls.c_t), st.c, "c_t")
    opt.close()


@pytest.mark.parametrize("bits", [2, 16])
def test_codec_all_zero_inputs(bits):
    """Zero blocks in the codec groups: scale 0, codes 0, errors 0."""
    n, W = 5000, 3
    g = ob.CodecGroup(n, W, bits, 256, period=1, seed=3, b1=0.9, b2=0.999, eps=1e-8, lr=1e-4)
    lay = O.Layout(n, W, 256, 256)
    st = O.State(lay)
    p0 = np.zeros(lay.n_pad, f32)
    p0[:n] = np.linspace(-1, 1, n, dtype=f32)
    st.p[:] = p0
    g.p.copy_(dev(p0))
    st.v[:n] = f32(1e-6)
    g.v[:n] = 1e-6
    zeros = [np.zeros(lay.n_pad, f32) for _ in range(W)]
    g.begin_compression()
    for t in range(1, 3):
        g.compressed_step([dev(z) for z in zeros])
        O.codec_step(st, zeros, dict(b1=0.9, b2=0.999, eps=1e-8, lr=1e-4), bits, t, 3, period=1)
    torch.cuda.synchronize()
    assert_bits_equal(host(g.p), st.p, "p")
    assert_bits_equal(host(g.m), st.m, "m")
    if bits != 16:
        assert np.all(host(g.bscales) == 0) and np.all(host(g.codes) == 0)
    g.close()
