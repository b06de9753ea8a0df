"""Parity of the layerwise mixed-width codecs (b-bit blocks with error
feedback, FP16 every period-th step) on the GPU, through the C ABI, with
the oracle, element by element, on the same seeded inputs.

Bar: codes, block scales and every float buffer bit-exact after each of
several consecutive steps (both sides round every operation the same way;
the quantizer's uniforms come from the same Philox counters; binary16
rounding is IEEE's).  NaN inputs are left out of the FP16 cases: the
binary16 bit pattern of a NaN is not fixed by IEEE.
"""
import numpy as np
import pytest
import torch

import momentum_compression_gb300 as ob
import oracle as O
import synth
from helpers import assert_bits_equal, bf16_tensor, dev, host

pytestmark = pytest.mark.gpu

f32 = np.float32
HP = dict(b1=0.9, b2=0.999, eps=1e-8, lr=1e-4)


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)
    from momentum_compression_gb300 import _build
    _build.build()
    yield
    torch.cuda.synchronize()


class Group:
    """One codec group on both sides: the GPU buffers and the oracle state,
    from the same host-drawn initial values."""

    def __init__(self, n, W, bits, A, dt, seed, clip=0.0):
        self.n, self.W, self.bits, self.dt = n, W, bits, dt
        self.hp = dict(HP, clip=clip)
        self.lay = O.Layout(n, W, A, A)
        self.opt = ob.CodecGroup(n, W, bits, A, dt, period=3, seed=seed, clip_value=clip, **HP)
        assert self.opt.n_pad == self.lay.n_pad
        self.rng = np.random.default_rng(seed + n + 7 * W + bits)
        self.st = O.State(self.lay)
        st, opt = self.st, self.opt
        st.m[:] = self.vec(1e-3)
        st.v[:] = np.abs(self.vec(1e-6)) + np.where(np.arange(self.lay.n_pad) < n, f32(1e-12), 0)
        st.p[:] = self.vec(0.02)
        for w in range(W):
            st.e[w][:] = self.vec(1e-4)
        st.e_s[:] = self.vec(1e-4)
        for name in ("m", "v", "p", "e_s"):
            getattr(opt, "err_s" if name == "e_s" else name).copy_(dev(getattr(st, name)))
        for w in range(W):
            opt.err[w].copy_(dev(st.e[w]))
        self.seed = seed

    def vec(self, scale):
        a = np.zeros(self.lay.n_pad, f32)
        a[: self.n] = self.rng.standard_normal(self.n).astype(f32) * f32(scale)
        return a

    def grads(self, scale=1e-3):
        g = [self.vec(scale) for _ in range(self.W)]
        if self.dt == "bf16":
            bits = [synth.bf16_bits(x) for x in g]
            return [synth.bf16_to_f32(b) for b in bits], [bf16_tensor(b) for b in bits]
        return g, [dev(x) for x in g]

    def step(self, t, scale=1e-3):
        gh, gd = self.grads(scale)
        self.opt.compressed_step(gd)
        O.codec_step(self.st, gh, self.hp, self.bits, t, self.seed + self.bits, period=3)
        torch.cuda.synchronize()

    def check(self, what):
        st, opt = self.st, self.opt
        assert_bits_equal(host(opt.m), st.m, f"{what}: m")
        assert_bits_equal(host(opt.p), st.p, f"{what}: p")
        assert_bits_equal(host(opt.err_s), st.e_s, f"{what}: e_s")
        for w in range(self.W):
            assert_bits_equal(host(opt.err[w]), st.e[w], f"{what}: e[{w}]")
        if self.bits == 16:
            if hasattr(st, "h"):
                assert_bits_equal(host(opt.h).view(np.uint16), st.h, f"{what}: h")
                assert_bits_equal(host(opt.hs).view(np.uint16), st.hs, f"{what}: hs")
        else:
            assert_bits_equal(host(opt.codes).view(np.uint32), st.codes, f"{what}: codes")
            assert_bits_equal(host(opt.bscales), st.bscales, f"{what}: bscales")
            assert_bits_equal(host(opt.scodes).view(np.uint32), st.scodes, f"{what}: scodes")
            assert_bits_equal(host(opt.sbscales), st.sbscales, f"{what}: sbscales")


# (n, W, bits, A, grad dtype)
QB_CASES = [
    (1, 1, 2, 256, "f32"),
    (255, 2, 2, 256, "f32"),
    (256, 3, 4, 256, "f32"),
    (4097, 2, 2, 256, "bf16"),
    (70_001, 8, 2, 4096, "f32"),        # several tiles per partition, ragged tail
    (70_001, 8, 4, 4096, "bf16"),
    (50_000, 5, 8, 512, "f32"),
    (300_000, 16, 2, 4096, "f32"),      # two batches of 8 workers in the server
    (9_000, 64, 2, 256, "f32"),         # the largest W
    (100, 4, 2, 4096, "f32"),           # partitions 1..3 are all padding
]


@pytest.mark.parametrize("n,W,bits,A,dt", QB_CASES,
                         ids=["n{}-W{}-b{}-A{}-{}".format(*c) for c in QB_CASES])
def test_qb_steps_match_oracle(n, W, bits, A, dt):
    g = Group(n, W, bits, A, dt, seed=1234)
    for t in range(1, 4):
        g.step(t)
        g.check(f"step {t}")


@pytest.mark.parametrize("n,W,dt", [(1, 1, "f32"), (4097, 3, "bf16"), (70_001, 8, "f32"),
                                    (100, 4, "f32")])
def test_f16_steps_match_oracle(n, W, dt):
    """Period 3: steps 1, 2 keep everything in the errors, step 3 sends."""
    g = Group(n, W, 16, 256, dt, seed=99)
    for t in range(1, 7):
        g.step(t)
        g.check(f"step {t}")
        if t % 3:
            assert torch.count_nonzero(g.opt.m).item() == 0


@pytest.mark.parametrize("bits", [2, 16])
def test_codecs_with_clip(bits):
    """The clamp of the compensated value ("1bit Adam" write-up 4.1) in the
    codec groups' worker kernels: large gradients so that it bites."""
    g = Group(20_000, 4, bits, 256, "f32", seed=5, clip=2e-3)
    for t in range(1, 4):
        g.step(t, scale=3e-3)
        g.check(f"step {t}")


def test_qb_nan_codes_zero_and_matches():
    """A NaN in a gradient: its code is 0 and the block's scale ignores it;
    its error is NaN on both sides."""
    g = Group(5000, 2, 2, 256, "f32", seed=3)
    gh, gd = g.grads()
    gh[0][100] = np.nan
    gd[0][100] = float("nan")
    g.opt.compressed_step(gd)
    O.codec_step(g.st, gh, g.hp, 2, 1, g.seed + 2, period=3)
    torch.cuda.synchronize()
    codes = host(g.opt.codes).view(np.uint32)
    assert_bits_equal(codes, g.st.codes, "codes")
    assert_bits_equal(host(g.opt.bscales), g.st.bscales, "bscales")
    e0 = host(g.opt.err[0])
    assert np.isnan(e0[100]) and np.isnan(g.st.e[0][100])
    ok = np.arange(g.lay.n_pad) != 100
    assert_bits_equal(e0[ok], g.st.e[0][ok], "e[0]")


def test_mixed_optimizer_matches_oracle():
    """Three groups (1, 2 and 16 bits) through warmup, the start of the
    compressed phase and 12 compressed steps (FP16 sent at steps 5 and 10),
    every buffer bit-exact after every step."""
    W, seed = 4, 1234
    specs = [(1, 5000, [0, 1000, 5000]), (2, 70_001, None), (16, 3000, None)]
    opt = ob.MixedOptimizer(specs, W, chunk=4096, period=5, seed=seed, **HP)
    rng = np.random.default_rng(17)
    ref = []
    for (bits, n, off), (_, g) in zip(specs, opt.groups):
        lay = O.Layout(n, W, 4096, 4096)
        st = O.State(lay, O.Layers(off) if off else None)
        st.p[:n] = rng.standard_normal(n).astype(f32) * f32(0.02)
        g.p.copy_(dev(st.p))
        ref.append((bits, lay, st))

    def draw():
        out_h, out_d = [], []
        for bits, lay, st in ref:
            gs = []
            for _ in range(W):
                a = np.zeros(lay.n_pad, f32)
                a[: lay.n] = rng.standard_normal(lay.n).astype(f32) * f32(1e-3)
                gs.append(a)
            out_h.append(gs)
            out_d.append([dev(a) for a in gs])
        return out_h, out_d

    for _ in range(3):
        gh, gd = draw()
        opt.warmup_step(gd)
        for (bits, lay, st), g in zip(ref, gh):
            O.warmup_step(lay, g, 0, HP, st.m, st.v, st.p, st.layers)
    opt.begin_compression()
    for bits, lay, st in ref:
        O.begin_compression(st, 3)
    for t in range(1, 13):
        gh, gd = draw()
        opt.compressed_step(gd)
        for (bits, lay, st), g in zip(ref, gh):
            O.codec_step(st, g, HP, bits, t, seed + bits, period=5)
        torch.cuda.synchronize()
        for (bits, lay, st), (_, g) in zip(ref, opt.groups):
            what = f"step {t}, {bits}-bit group"
            assert_bits_equal(host(g.p), st.p, f"{what}: p")
            if bits != 1:  # the 1-bit group's m and errors are in deferred form
                assert_bits_equal(host(g.m), st.m, f"{what}: m")
                assert_bits_equal(host(g.err_s), st.e_s, f"{what}: e_s")
    opt.close()


def _torch_state(g, n, seed):
    """m ~ N(0, 1e-3), v ~ |N(0, 1e-6)| + 1e-12, p ~ N(0, 0.02), errors
    ~ N(0, 1e-4), drawn on the GPU by torch's seeded generator (padding 0)."""
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    r = lambda s: torch.randn(n, generator=gen, device="cuda") * s
    g.m[:n] = r(1e-3)
    g.v[:n] = r(1e-6).abs() + 1e-12
    g.p[:n] = r(0.02)
    for e in g.err:
        e[:n] = r(1e-4)
    g.err_s[:n] = r(1e-4)


@pytest.mark.slow
def test_resnet50_mixed_full_size():
    """The ResNet-50 mixed workload at W = 8 in bench.py's configuration.
    2-bit group (23.5 M elements): one step on the GPU, the oracle on
    sampled blocks of 256 -- a block's step reads only its own elements of
    every worker, the server and the update -- the first, one in the
    middle, the last real one and one of the padding tail.  FP16 group
    (53 k elements): a sending step, checked whole."""
    groups = synth.mixed_groups(W=8)
    W = 8
    specs = [(bits, wl.n, wl.layer_offsets) for bits, wl in groups]
    opt = ob.MixedOptimizer(specs, W, chunk=1 << 20, period=synth.NORM_PERIOD, seed=1234,
                            **synth.ADAM_HP)
    gens = {}
    for (bits, wl), (_, g) in zip(groups, opt.groups):
        if bits == 1:
            continue
        _torch_state(g, wl.n, 77 + bits)
        gen = torch.Generator(device="cuda")
        gen.manual_seed(synth.SEED_BASE + bits)
        sizes = torch.tensor([s for _, s, _ in wl.tensors], device="cuda")
        std = torch.zeros(g.n_pad, device="cuda")
        std[: wl.n] = torch.repeat_interleave(
            torch.tensor(wl.layer_std, dtype=torch.float32, device="cuda"), sizes)
        gens[bits] = [torch.randn(g.n_pad, generator=gen, device="cuda") * std for _ in range(W)]
    hp = dict(synth.ADAM_HP)

    # 2-bit group: sampled blocks
    wl2, g2 = dict(groups)[2], dict(opt.groups)[2]
    lay2 = O.Layout(wl2.n, W, 4096, 4096)
    assert lay2.n_pad == g2.n_pad
    nblk = g2.n_pad // 256
    picks = sorted({0, nblk // 2, (wl2.n - 1) // 256, nblk - 1})
    before = {}
    for b in picks:
        s = slice(256 * b, 256 * b + 256)
        before[b] = dict(m=host(g2.m[s]).copy(), v=host(g2.v[s]).copy(), p=host(g2.p[s]).copy(),
                         e_s=host(g2.err_s[s]).copy(),
                         e=[host(e[s]).copy() for e in g2.err],
                         g=[host(x[s]).copy() for x in gens[2]])
    # FP16 group: whole, a sending step (t = 10)
    wl16, g16 = dict(groups)[16], dict(opt.groups)[16]
    lay16 = O.Layout(wl16.n, W, 4096, 4096)
    st16 = O.State(lay16)
    st16.m[:], st16.v[:], st16.p[:] = host(g16.m), host(g16.v), host(g16.p)
    st16.e_s[:] = host(g16.err_s)
    for w in range(W):
        st16.e[w][:] = host(g16.err[w])
    g16h = [host(x).copy() for x in gens[16]]

    g2.compressed_step(gens[2])
    g16.t = 9
    g16.compressed_step(gens[16])
    torch.cuda.synchronize()

    for b, d in before.items():
        s = slice(256 * b, 256 * b + 256)
        k0 = 256 * b
        codes, scs = [], []
        for w in range(W):
            c, sc = O.qb_compress_worker(lay2, 2, d["g"][w], d["m"], d["e"][w], hp["b1"], w,
                                         g2.key, 1, k0=k0, length=256)
            codes.append(c)
            scs.append(sc)
            assert_bits_equal(host(g2.codes[w, 16 * b: 16 * b + 16]).view(np.uint32), c,
                              f"block {b} codes of worker {w}")
            assert_bits_equal(host(g2.bscales[w, b: b + 1]), sc, f"block {b} scale {w}")
            assert_bits_equal(host(g2.err[w][s]), d["e"][w], f"block {b} e[{w}]")
        sc_, ss_ = O.qb_server(lay2, 2, np.stack(codes), np.stack(scs), d["e_s"], g2.key, 1,
                               k0=k0, length=256)
        assert_bits_equal(host(g2.scodes[16 * b: 16 * b + 16]).view(np.uint32), sc_,
                          f"block {b} server codes")
        assert_bits_equal(host(g2.sbscales[b: b + 1]), ss_, f"block {b} server scale")
        assert_bits_equal(host(g2.err_s[s]), d["e_s"], f"block {b} e_s")
        m, p = d["m"].copy(), d["p"].copy()
        O.qb_adam(lay2, 2, sc_, ss_, d["v"], hp["eps"], hp["lr"], m, p, k0=k0, length=256)
        assert_bits_equal(host(g2.m[s]), m, f"block {b} m")
        assert_bits_equal(host(g2.p[s]), p, f"block {b} p")

    O.codec_step(st16, g16h, hp, 16, 10, g16.key, period=synth.NORM_PERIOD)
    assert_bits_equal(host(g16.p), st16.p, "FP16 group p")
    assert_bits_equal(host(g16.m), st16.m, "FP16 group m")
    assert_bits_equal(host(g16.err_s), st16.e_s, "FP16 group e_s")
    for w in range(W):
        assert_bits_equal(host(g16.err[w]), st16.e[w], f"FP16 group e[{w}]")
    opt.close()
