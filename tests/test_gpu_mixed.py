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
        O.codec_step(self.st, gh, self.hp, self.bits, t, self.seed, period=3)
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
    O.codec_step(g.st, gh, g.hp, 2, 1, g.seed, period=3)
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
