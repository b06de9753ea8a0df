"""Pins for the oracle: each test checks oracle/ against something other
than itself -- hand-computed worked examples (tests/golden/), closed forms,
invariants the pages state, brute force in float64, and independent
libraries (curand's host Philox generator, torch.optim.Adam).

No GPU is needed; these run in the CPU suite.
"""
import ctypes as ct
import glob
import json
import math
import os

import numpy as np
import pytest

import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")
f32 = np.float32


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def _eq(a, b):
    a = np.asarray(a, np.float32)
    b = np.asarray(b, np.float32)
    assert a.shape == b.shape
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), (a, b)


# ---------------------------------------------------------------------------
# Hand-computed worked examples
# ---------------------------------------------------------------------------

def test_worked_example_adam():
    G = _load("worked_example_adam.json")
    i, x = G["inputs"], G["expected"]
    lay = O.Layout(i["n"], i["W"], i["A"], i["C"])
    assert (lay.P, lay.n_pad, lay.cpp, lay.nc) == (2, 4, 1, 2)
    m = np.zeros(4, f32)
    e = [np.zeros(4, f32) for _ in range(2)]
    bits = np.zeros((2, lay.words), np.uint32)
    scales = np.zeros((2, lay.nc), f32)
    for w in range(2):
        b, s, _ = O.compress_worker(lay, np.array(i["g"][w], f32), m, e[w], i["b1"])
        bits[w], scales[w] = b, s
        _eq(s, x["scales"][w])
        assert int(b[0]) == x["bits"][w]
        _eq(e[w], x["e"][w])
    e_s = np.zeros(4, f32)
    sbits, sscales, y = O.server_reduce(lay, bits, scales, e_s)
    _eq(y, x["y"])
    _eq(sscales, x["sscales"])
    assert int(sbits[0]) == x["sbits"]
    _eq(e_s, x["e_s"])
    p = np.zeros(4, f32)
    O.adam_update(lay, sbits, sscales, np.array(i["v_frozen"], f32), i["eps"],
                  i["lr"], m, p)
    _eq(m, x["m"])
    _eq(p, x["p"])
    _eq(O.decompress(lay, sbits, sscales), x["m"])
    # the error monitor on the same step, by hand: per chunk the sum of the
    # squared errors, e_0 = [-0.5,-0.5 | 1.5,-1.5] -> [0.5, 4.5],
    # e_1 = [0.5,-0.5 | 0,0] -> [0.5, 0], e_s = [0.75,-0.75 | 0,0] -> [1.125, 0]
    _eq(O.error_norm(lay, e[0]), [0.5, 4.5])
    _eq(O.error_norm(lay, e[1]), [0.5, 0.0])
    _eq(O.error_norm(lay, e_s), [1.125, 0.0])


def test_error_norm_against_fp64_and_padding():
    """Random errors over a layout with ragged chunks and a padding tail:
    each chunk's value is within the fp32 summation bound of the fp64 sum
    of squares of its real elements, and whatever sits in the padding
    changes nothing."""
    rng = np.random.default_rng(41)
    n, W, A, C = 30_001, 3, 4096, 3000
    lay = O.Layout(n, W, A, C)
    e = np.zeros(lay.n_pad, f32)
    e[:n] = rng.standard_normal(n).astype(f32) * f32(1e-3)
    got = O.error_norm(lay, e)
    assert got.shape == (lay.nc,)
    for g in range(lay.nc):
        s, ln, real = lay.chunk_range(g)
        want = float(np.sum(e[s:s + real].astype(np.float64) ** 2))
        assert abs(float(got[g]) - want) <= (real + 2) * 2.0 ** -23 * want + 1e-45, g
        if real == 0:
            assert got[g] == 0.0
    junk = e.copy()
    junk[n:] = f32(1e30)
    _eq(O.error_norm(lay, junk), got)


def test_worked_example_lamb():
    G = _load("worked_example_lamb.json")
    i, x = G["inputs"], G["expected"]
    lay = O.Layout(i["n"], i["W"], i["A"], i["C"])
    layers = O.Layers(i["layer_offsets"])
    ls = {"s": np.array(i["s"], f32), "c_avg": np.array(i["c_avg"], f32),
          "r_prev": np.ones(2, f32), "c_prev": np.array(i["c_avg"], f32),
          "c_prev2": np.array(i["c_avg"], f32)}
    rho = O.rho_of(ls)
    _eq(rho, [1.0, 1.0])
    m = np.zeros(4, f32)
    e = [np.zeros(4, f32) for _ in range(2)]
    bits = np.zeros((2, lay.words), np.uint32)
    scales = np.zeros((2, lay.nc), f32)
    for w in range(2):
        b, s, _ = O.compress_worker(lay, np.array(i["g"][w], f32), m, e[w], i["b1"],
                                    layers, ls["s"], rho)
        bits[w], scales[w] = b, s
        _eq(s, x["scales"][w])
        assert int(b[0]) == x["bits"][w]
        _eq(e[w], x["e"][w])
    e_s = np.zeros(4, f32)
    sbits, sscales, _ = O.server_reduce(lay, bits, scales, e_s, layers, rho)
    _eq(sscales, x["sscales"])
    assert int(sbits[0]) == x["sbits"]
    _eq(e_s, x["e_s"])
    vf = np.array(i["v_frozen"], f32)
    v_fresh = vf.copy()
    R = O.lamb_pass_a(lay, layers, ls["s"], sbits, sscales, vf, i["b1"], i["b2"],
                      m, v_fresh)
    _eq(m, x["m"])
    _eq(v_fresh, x["v_fresh"])
    _eq(R[0], np.float32(4.0) / np.float32(2.5))
    _eq(R[1], x["R_layer1"])
    c = O.lamb_ratio(R, i, ls)
    _eq(ls["r_prev"], x["r"])
    _eq(c, x["c"])
    _eq(ls["c_prev"], x["c"])
    _eq(ls["c_prev2"], x["c_prev2"])
    p = np.zeros(4, f32)
    O.lamb_pass_b(lay, layers, c, m, vf, i["eps"], i["lr"], p)
    _eq(p, x["p"])
    _eq(O.decompress(lay, sbits, sscales, layers, ls["s"]), x["m"])


# ---------------------------------------------------------------------------
# Canonical reduction
# ---------------------------------------------------------------------------

def test_cr_canonical_order_hand_value():
    """One tile: a[0] = 2^24 and a[4p] = 1 for p = 1..255.  Lane 0 holds
    2^24, lanes 1..255 hold 1.  In warp 0 the first butterfly step loses
    one unit (2^24 + 1 rounds to 2^24), every later sum is exact: warp 0 =
    2^24 + 30, warps 1..7 = 32, total 2^24 + 254.  A plain sequential sum
    would give 2^24, the exact sum 2^24 + 255."""
    a = np.zeros(4096, f32)
    a[0] = 2.0 ** 24
    a[4 * np.arange(1, 256)] = 1.0
    assert O.cr_sum(a) == f32(2 ** 24 + 254)


def test_cr_tiles_summed_in_order():
    """Tile totals 2^24, 1, 1 summed left to right: each +1 is lost."""
    a = np.zeros(3 * 4096, f32)
    a[0], a[4096], a[8192] = 2.0 ** 24, 1.0, 1.0
    assert O.cr_sum(a) == f32(2 ** 24)
    # ... while inside one lane the same values add up in element order:
    b = np.zeros(4096, f32)
    b[0], b[1], b[2] = 1.0, 1.0, 2.0 ** 24
    assert O.cr_sum(b) == f32(2 ** 24 + 2)


def test_cr_warp_sums_paired_in_order():
    """The 8 warp sums of a tile are added as ((w0+w1)+(w2+w3)) + ...: with
    w0 = 2^24, w1 = 1, w2 = -2^24, w3 = 1 (one element per warp, at lane
    32w) this gives 2^24 + (-2^24 + 1) = 1, where (w0+w2)+(w1+w3) would
    give 2."""
    a = np.zeros(4096, f32)
    a[0], a[128], a[256], a[384] = 2.0 ** 24, 1.0, -(2.0 ** 24), 1.0
    assert O.cr_sum(a) == f32(1.0)


@pytest.mark.parametrize("count", [0, 1, 3, 4, 5, 1023, 1024, 4095, 4096, 4097,
                                   12289, 70000])
def test_cr_integers_exact(count):
    rng = np.random.default_rng(count)
    a = rng.integers(0, 100, size=count).astype(f32)
    assert O.cr_sum(a) == f32(a.astype(np.int64).sum())


def test_cr_close_to_exact_sum():
    rng = np.random.default_rng(5)
    for count in (17, 4096, 50000, 300001):
        a = np.abs(rng.standard_normal(count)).astype(f32)
        exact = a.astype(np.float64).sum()
        # error bound of any summation order: (count-1) * u * sum|a|
        bound = (count - 1) * 2.0 ** -24 * exact
        assert abs(float(O.cr_sum(a)) - exact) <= bound


# ---------------------------------------------------------------------------
# Layout
# ---------------------------------------------------------------------------

def test_layout():
    lay = O.Layout(1 << 20, 4, 4096, 1 << 18)
    assert (lay.P, lay.n_pad, lay.cpp, lay.nc) == (1 << 18, 1 << 20, 1, 4)
    lay = O.Layout(109482240, 8, 4096, 1 << 20)
    assert lay.P == 13688832 and lay.n_pad == 8 * 13688832
    assert lay.cpp == 14 and lay.chunk_range(13) == (13 * (1 << 20), 57344, 57344)
    lay = O.Layout(100, 4, 4096, 1 << 20)      # partitions 1..3 are all padding
    assert lay.P == 4096 and lay.C == 4096 and lay.chunk_range(1)[2] == 0
    lay = O.Layout(5000, 3, 32, 1000)
    assert lay.P == 1696 and lay.cpp == 2 and lay.chunk_range(1) == (1000, 696, 696)
    assert lay.chunk_range(5) == (4392, 696, 608)


# ---------------------------------------------------------------------------
# Compressor invariants (I1-I4)
# ---------------------------------------------------------------------------

def _rand_case(n=5000, W=3, A=32, C=1000, seed=0):
    rng = np.random.default_rng(seed)
    lay = O.Layout(n, W, A, C)
    g = [np.zeros(lay.n_pad, f32) for _ in range(W)]
    for w in range(W):
        g[w][:n] = rng.standard_normal(n).astype(f32) * f32(1e-3)
    m = np.zeros(lay.n_pad, f32)
    m[:n] = rng.standard_normal(n).astype(f32) * f32(1e-3)
    e = [np.zeros(lay.n_pad, f32) for _ in range(W)]
    for w in range(W):
        e[w][:n] = rng.standard_normal(n).astype(f32) * f32(1e-4)
    return lay, g, m, e


def _bits_of(words, n_pad):
    return np.unpackbits(words.view(np.uint8), bitorder="little")[:n_pad].astype(bool)


def test_compress_invariants():
    lay, g, m, e = _rand_case()
    n = lay.n
    e0 = e[0].copy()
    bits, scales, x = O.compress_worker(lay, g[0], m, e[0], 0.9)
    # x follows the momentum recurrence and adds the carried error
    xb = ((f32(0.9) * m[:n]) + (f32(1) - f32(0.9)) * g[0][:n]) + e0[:n]
    _eq(x[:n], xb)
    b = _bits_of(bits, lay.n_pad)
    # I2/I3: bit k of word k/32 (LSB first) is x >= 0; padding bits 0
    assert np.array_equal(b[:n], x[:n] >= 0)
    assert not b[n:].any()
    # I1: x == scale*sign(x) + e' within 1 ulp
    for gi in range(lay.nc):
        s, ln, real = lay.chunk_range(gi)
        if real == 0:
            assert scales[gi] == 0
            continue
        xs = x[s:s + real].astype(np.float64)
        sg = np.where(x[s:s + real] >= 0, 1.0, -1.0)
        rec = scales[gi] * sg + e[0][s:s + real].astype(np.float64)
        # e' = fl(x - scale*sign) is rounded once, relative to the larger of
        # |x| and |e'|
        big = np.maximum(np.abs(x[s:s + real]), np.abs(e[0][s:s + real]))
        ulp = np.spacing(big.astype(f32)).astype(np.float64)
        assert np.all(np.abs(rec - xs) <= ulp)
        # I4: scale is mean |x| over the chunk's real elements (fp64 bound)
        mean = np.abs(xs).mean()
        assert abs(scales[gi] - mean) <= (real + 1) * 2.0 ** -24 * mean
    assert np.all(e[0][n:] == 0)


def test_sign_of_zero_and_nan():
    lay = O.Layout(64, 1, 32, 64)
    g = np.zeros(64, f32)
    m = np.zeros(64, f32)
    e = np.zeros(64, f32)
    g[1] = -0.0
    e[2] = -0.0
    g[3] = np.nan
    g[4:] = 1.0
    g[5] = -1.0
    bits, scales, x = O.compress_worker(lay, g, m, e, 0.5)
    b = _bits_of(bits, 64)
    assert b[0] and b[1] and b[2]       # +0 and -0 pack as +1
    assert not b[3]                      # NaN packs as -1
    assert b[4] and not b[5]


def test_lsb_first_single_negative():
    for k in (0, 1, 31, 32, 33, 63):
        lay = O.Layout(64, 1, 32, 64)
        g = np.ones(64, f32)
        g[k] = -1.0
        bits, _, _ = O.compress_worker(lay, g, np.zeros(64, f32), np.zeros(64, f32), 0.0)
        expect = np.array([0xFFFFFFFF, 0xFFFFFFFF], np.uint32)
        expect[k // 32] ^= np.uint32(1 << (k % 32))
        assert np.array_equal(bits, expect)


def test_constant_magnitude_is_lossless():
    """Scaled sign is exact when every |x| in a chunk is equal: the error is
    0 and the decompressed value is x itself; the server then passes the
    worker average through unchanged."""
    lay = O.Layout(256, 2, 32, 64)
    g0 = np.where(np.arange(256) % 3 == 0, 4.0, -4.0).astype(f32)
    g1 = g0.copy()
    m = np.zeros(256, f32)
    e = [np.zeros(256, f32), np.zeros(256, f32)]
    bits, scales = np.zeros((2, lay.words), np.uint32), np.zeros((2, lay.nc), f32)
    for w, g in enumerate((g0, g1)):
        b, s, x = O.compress_worker(lay, g, m, e[w], 0.5)
        bits[w], scales[w] = b, s
        assert np.all(e[w] == 0) and np.all(s == 2.0)
    e_s = np.zeros(256, f32)
    sbits, sscales, y = O.server_reduce(lay, bits, scales, e_s)
    assert np.all(e_s == 0)
    _eq(O.decompress(lay, sbits, sscales), 0.5 * g0)


def test_server_matches_float64_average():
    lay, g, m, e = _rand_case(n=3000, W=4, A=32, C=512, seed=3)
    bits = np.zeros((lay.W, lay.words), np.uint32)
    scales = np.zeros((lay.W, lay.nc), f32)
    xs = []
    for w in range(lay.W):
        b, s, x = O.compress_worker(lay, g[w], m, e[w], 0.9)
        bits[w], scales[w] = b, s
        xs.append(x)
    rng = np.random.default_rng(9)
    e_s = np.zeros(lay.n_pad, f32)
    e_s[:lay.n] = rng.standard_normal(lay.n).astype(f32) * f32(1e-4)
    e_s0 = e_s.copy()
    sbits, sscales, y = O.server_reduce(lay, bits, scales, e_s)
    n = lay.n
    dec = np.zeros((lay.W, n))
    for w in range(lay.W):
        sg = np.where(_bits_of(bits[w], lay.n_pad)[:n], 1.0, -1.0)
        ch = np.array([_chunk_of(lay, k) for k in range(n)])
        dec[w] = scales[w][ch] * sg
    z = dec.mean(axis=0)
    y64 = e_s0[:n].astype(np.float64) + z
    # W-1 additions, a division and one more addition, each rounded once:
    # at most (W+1) units of the magnitudes that were added
    mag = np.abs(dec).mean(axis=0) + np.abs(e_s0[:n])
    assert np.all(np.abs(y[:n] - y64) <= (lay.W + 1) * 2.0 ** -24 * mag)
    assert np.array_equal(_bits_of(sbits, lay.n_pad)[:n], y[:n] >= 0)


def _chunk_of(lay, k):
    j, r = divmod(k, lay.P)
    return j * lay.cpp + r // lay.C


# ---------------------------------------------------------------------------
# I5: the global-momentum identity of the 1-bit LAMB summary (paragraph 3),
#   m_t = b1*m_{t-1} + (1-b1)*g_bar_t + rho*delta~_{t-1} - delta~_t,
#   delta~ = (1/W) sum_i e_i + e_s,
# which with rho = 1 (1-bit Adam) telescopes to the error-feedback claim
# that the compressed sum tracks the true sum (lqnn.cn write-up, 2.1).
# ---------------------------------------------------------------------------

def _delta(st):
    return np.mean([e.astype(np.float64) for e in st.e], axis=0) + st.e_s


def test_i5_adam_identity_over_steps():
    n, W = 6000, 3
    lay = O.Layout(n, W, 32, 1024)
    st = O.State(lay)
    rng = np.random.default_rng(11)
    st.v[:n] = np.abs(rng.standard_normal(n)).astype(f32) * f32(1e-6) + f32(1e-8)
    st.m[:n] = rng.standard_normal(n).astype(f32) * f32(1e-3)
    hp = dict(b1=0.9, b2=0.999, eps=1e-8, lr=1e-4)
    d_prev = _delta(st)
    total_g = np.zeros(n)
    for t in range(10):
        g = [np.zeros(lay.n_pad, f32) for _ in range(W)]
        for w in range(W):
            g[w][:n] = rng.standard_normal(n).astype(f32) * f32(1e-3)
        gbar = np.mean([x.astype(np.float64) for x in g], axis=0)
        m_prev = st.m.astype(np.float64)
        O.compressed_step(st, g, hp)
        d = _delta(st)
        rhs = 0.9 * m_prev + 0.1 * gbar + d_prev - d
        scale = np.abs(m_prev).max() + np.abs(d).max()
        assert np.max(np.abs(st.m[:n] - rhs[:n])) <= 64 * 2.0 ** -24 * scale
        d_prev = d
        total_g += gbar[:n]


def test_i5_lamb_identity_scaled_space():
    """For 1-bit LAMB the identity holds for the scaled momentum sigma*m with
    rho = c_{t-2}/c_{t-1} on both the worker and the server error."""
    n, W = 5000, 2
    off = [0, 1000, 1003, 4096, 5000]
    lay = O.Layout(n, W, 32, 512)
    layers = O.Layers(off)
    st = O.State(lay, layers, lamb=True)
    rng = np.random.default_rng(12)
    st.v[:n] = np.abs(rng.standard_normal(n)).astype(f32) * f32(1e-6) + f32(1e-8)
    st.m[:n] = rng.standard_normal(n).astype(f32) * f32(1e-3)
    st.v_fresh[:] = st.v
    st.ls = {"s": np.array([1.0, 4.0, 0.5, 2.0], f32),
             "c_avg": np.array([1.0, 2.0, 0.5, 1.5], f32),
             "r_prev": np.ones(4, f32),
             "c_prev": np.array([1.0, 2.0, 0.5, 1.5], f32),
             "c_prev2": np.array([1.0, 2.0, 0.5, 1.5], f32)}
    hp = dict(b1=0.9, b2=0.999, eps=1e-6, lr=1e-3, r_thr=0.1, r_min=0.5,
              r_max=4.0, c_min=0.01, c_max=10.0)
    sig = np.repeat(st.ls["s"], np.diff(off)).astype(np.float64)
    d_prev = _delta(st)[:n]
    for t in range(6):
        rho = np.repeat(O.rho_of(st.ls), np.diff(off)).astype(np.float64)
        g = [np.zeros(lay.n_pad, f32) for _ in range(W)]
        for w in range(W):
            g[w][:n] = rng.standard_normal(n).astype(f32) * f32(1e-3 * 0.7 ** t)
        gbar = np.mean([x.astype(np.float64)[:n] for x in g], axis=0)
        m_prev = st.m[:n].astype(np.float64)
        O.compressed_step(st, g, hp, lamb=True)
        d = _delta(st)[:n]
        lhs = sig * st.m[:n]
        rhs = sig * (0.9 * m_prev + 0.1 * gbar) + rho * d_prev - d
        scale = np.abs(sig * m_prev).max() + np.abs(d).max() + np.abs(d_prev).max()
        assert np.max(np.abs(lhs - rhs)) <= 64 * 2.0 ** -24 * scale
        d_prev = d
    # rho really moved away from 1 during these steps
    assert np.any(O.rho_of(st.ls) != 1.0)


# ---------------------------------------------------------------------------
# I6: the r_t clip of the 1-bit LAMB summary, paragraph 1
# ---------------------------------------------------------------------------

def _ratio(R, r_prev, hp, c_avg=1.0):
    ls = {"c_avg": np.array([c_avg], f32), "r_prev": np.array([r_prev], f32),
          "c_prev": np.array([c_avg], f32), "c_prev2": np.array([c_avg], f32)}
    c = O.lamb_ratio(np.array([R], f32), hp, ls)
    return float(ls["r_prev"][0]), float(c[0]), ls


HP_L = dict(r_thr=0.1, r_min=0.5, r_max=4.0, c_min=0.01, c_max=10.0)


def test_i6_examples():
    assert _ratio(3.0, 1.0, HP_L)[0] == pytest.approx(1.1, abs=1e-7)
    assert _ratio(0.2, 1.0, HP_L)[0] == pytest.approx(0.9, abs=1e-7)
    assert _ratio(1.05, 1.0, HP_L)[0] == f32(1.05)
    assert _ratio(np.inf, 1.0, HP_L)[0] == pytest.approx(1.1, abs=1e-7)
    # sustained large ratios grow r by 1.1x per step until r_max = 4 holds
    r, steps = 1.0, 0
    while r < 4.0:
        r = _ratio(100.0, r, HP_L)[0]
        steps += 1
    assert r == 4.0 and 15 <= steps <= 16
    # c = clip(c_avg * r, c_min, c_max)
    assert _ratio(1.0, 1.0, HP_L, c_avg=20.0)[1] == 10.0
    assert _ratio(1.0, 1.0, HP_L, c_avg=1e-3)[1] == pytest.approx(0.01)


def test_i6_bounds_random():
    rng = np.random.default_rng(4)
    for _ in range(2000):
        r_prev = float(rng.uniform(0.5, 4.0))
        R = float(10 ** rng.uniform(-2, 2))
        r, _, _ = _ratio(R, r_prev, HP_L)
        lo, hi = (1 - 0.1) * r_prev, (1 + 0.1) * r_prev
        if max(lo, 0.5) <= min(hi, 4.0):
            assert max(lo, 0.5) * (1 - 1e-6) <= r <= min(hi, 4.0) * (1 + 1e-6)
        else:
            assert 0.5 <= r <= 4.0


def test_lamb_frozen_is_basic_one_bit():
    r, c, ls = _ratio(3.0, 1.0, HP_L, c_avg=2.5)
    ls2 = {"c_avg": np.array([2.5], f32), "r_prev": np.ones(1, f32),
           "c_prev": np.array([2.5], f32), "c_prev2": np.array([2.5], f32)}
    c2 = O.lamb_ratio(np.array([3.0], f32), HP_L, ls2, frozen=True)
    assert c2[0] == 2.5 and ls2["r_prev"][0] == 1.0


def test_lamb_lossless_reconstructs_gradient():
    """When compression is lossless (constant |x| per chunk, zero errors)
    the reconstructed gradient of pass A is the averaged gradient itself."""
    n = 128
    lay = O.Layout(n, 1, 32, 32)
    layers = O.Layers([0, 64, 128])
    ls = {"s": np.array([2.0, 0.5], f32)}
    g = np.where(np.arange(n) % 5 < 2, 3.0, -3.0).astype(f32)
    m_prev = np.zeros(n, f32)
    e = np.zeros(n, f32)
    b, s, x = O.compress_worker(lay, g, m_prev, e, 0.5, layers, ls["s"])
    assert np.all(e == 0)
    e_s = np.zeros(n, f32)
    sb, ss, _ = O.server_reduce(lay, b[None], s[None], e_s, layers)
    assert np.all(e_s == 0)
    m = m_prev.copy()
    vf = np.ones(n, f32)
    vt = vf.copy()
    O.lamb_pass_a(lay, layers, ls["s"], sb, ss, vf, 0.5, 0.5, m, vt)
    _eq(m, 0.5 * g)                     # m_t = (1-b1) g
    _eq(vt, 0.5 * 1.0 + 0.5 * g * g)   # v_t = b2 v + (1-b2) g^2 with g recovered


@pytest.mark.parametrize("lamb", [False, True])
def test_stored_momentum_is_the_scaled_signs(lamb):
    """After every compressed step the stored momentum is exactly the
    server's chunk scale times its sign ([LAMB] 1-2: m_t = M/sigma_l for
    LAMB, sscale*sign for Adam), element by element -- recomputed here in
    NumPy from the server output, with one IEEE division per element.  This
    is what lets the momentum be held in sign form between steps.  Odd
    layer sizes, W = 3, padding, 4 steps with a falling gradient scale."""
    sizes = [7, 1, 4095, 33, 3000]
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.uint64)
    n, W = int(off[-1]), 3
    lay = O.Layout(n, W, 32, 1024)
    layers = O.Layers(off) if lamb else O.Layers()
    st = O.State(lay, layers, lamb=lamb)
    rng = np.random.default_rng(5)
    st.v[:n] = np.abs(rng.standard_normal(n)).astype(f32) * f32(1e-6) + f32(1e-12)
    st.m[:n] = rng.standard_normal(n).astype(f32) * f32(1e-3)
    st.p[:n] = rng.standard_normal(n).astype(f32) * f32(0.02)
    hp = dict(b1=0.9, b2=0.999, eps=1e-6, lr=1e-3, r_thr=0.1, r_min=0.5, r_max=4.0,
              c_min=0.01, c_max=10.0)
    L = len(sizes)
    if lamb:
        st.v_fresh[:] = st.v
        st.ls = {"s": (10.0 ** rng.uniform(-1, 1, L)).astype(f32),
                 "c_avg": np.ones(L, f32), "r_prev": np.ones(L, f32),
                 "c_prev": np.ones(L, f32), "c_prev2": np.ones(L, f32)}
    # per element: its chunk's index and (LAMB) its layer's sigma
    chunk_of = np.zeros(lay.n_pad, np.int64)
    for g in range(lay.nc):
        s0, ln, _ = lay.chunk_range(g)
        chunk_of[s0:s0 + ln] = g
    sigma = (np.repeat(st.ls["s"], sizes) if lamb else np.ones(n, f32)).astype(f32)
    for t in range(4):
        grads = []
        for w in range(W):
            a = np.zeros(lay.n_pad, f32)
            a[:n] = rng.standard_normal(n).astype(f32) * f32(1e-3 * 3.0 ** -t)
            grads.append(a)
        O.compressed_step(st, grads, hp, lamb=lamb)
        k = np.arange(n)
        bit = (st.sbits[k >> 5] >> (k & 31).astype(np.uint32)) & 1
        M = st.sscales[chunk_of[:n]] * np.where(bit == 1, f32(1), f32(-1))
        want = (M / sigma).astype(f32) if lamb else M.astype(f32)
        _eq(st.m[:n], want)
        assert not st.m[n:].any()


def test_adam_update_hand_with_eps():
    """[LAMB] ¶1 / [BLOG] §2.1 with eps > 0, by hand (dyadic values):
    m = sscale*sign = [1.25, -1.25]; d = sqrt(v) + eps = [2 + 0.5, 0.5 + 0.5];
    u = m/d = [0.5, -1.25]; p = 0 - lr*u with lr = 0.5."""
    lay = O.Layout(2, 1, 1, 2)
    sbits = np.array([0b01], np.uint32)
    sscales = np.array([1.25], f32)
    v = np.array([4.0, 0.25], f32)
    m = np.zeros(2, f32)
    p = np.zeros(2, f32)
    O.adam_update(lay, sbits, sscales, v, 0.5, 0.5, m, p)
    _eq(m, [1.25, -1.25])
    _eq(p, [-0.25, 0.625])


def test_compress_momentum_with_b1_not_half():
    """[BLOG] §2.1, m_w = b1*m + (1-b1)*g, with b1 = 0.75 so that b1 and
    1 - b1 differ (the worked examples use 0.5), by hand:
    m_w = [0.75 + 0.5, -1.5 + 1] = [1.25, -0.5]; scale = 0.875; bits 0b01;
    e' = x - scale*sign = [0.375, 0.375]."""
    lay = O.Layout(2, 1, 1, 2)
    e = np.zeros(2, f32)
    b, s, x = O.compress_worker(lay, np.array([2.0, 4.0], f32), np.array([1.0, -2.0], f32),
                                e, 0.75)
    _eq(x, [1.25, -0.5])
    _eq(s, [0.875])
    assert int(b[0]) == 0b01
    _eq(e, [0.375, 0.375])


def test_rho_is_the_ratio_of_the_two_previous_coefficients():
    """[LAMB] ¶3: the error is scaled by rho = c_{t-2}/c_{t-1}."""
    _eq(O.rho_of({"c_prev2": np.array([3.0, 1.0], f32), "c_prev": np.array([2.0, 4.0], f32)}),
        [1.5, 0.25])


def test_lamb_pass_a_hand_with_b2_not_half():
    """[LAMB] ¶1 pass A with b1 = 0.5 and b2 = 0.75 (b2 and 1 - b2 differ), by
    hand: M = [1, -1] (sigma 1) = m_t; g = (m_t - 0.5*[0.5, 0.5])/0.5 =
    [1.5, -2.5]; v_t = 0.75*[1, 4] + 0.25*g^2 = [1.3125, 4.5625];
    R = max(v_Tw / v_t) with v_Tw = [2.625, 4.5625] = 2."""
    lay = O.Layout(2, 1, 1, 2)
    layers = O.Layers([0, 2])
    m = np.array([0.5, 0.5], f32)
    vt = np.array([1.0, 4.0], f32)
    R = O.lamb_pass_a(lay, layers, np.array([1.0], f32), np.array([0b01], np.uint32),
                      np.array([1.0], f32), np.array([2.625, 4.5625], f32), 0.5, 0.75, m, vt)
    _eq(m, [1.0, -1.0])
    _eq(vt, [1.3125, 4.5625])
    _eq(R, [2.0])


def test_lamb_ratio_shifts_the_coefficient_history():
    """After a LAMB step c_{t-2} <- c_{t-1} <- c_t and r_prev <- r_t
    ([LAMB] ¶1, ¶3): with c_prev = 5 and c_prev2 = 7, c_prev2 becomes 5.
    R = 3 is clipped to (1 + r_thr)*r_prev; c = c_avg*r."""
    hp = dict(r_thr=0.1, r_min=0.5, r_max=4.0, c_min=0.01, c_max=10.0)
    ls = {"c_avg": np.array([2.0], f32), "r_prev": np.array([1.0], f32),
          "c_prev": np.array([5.0], f32), "c_prev2": np.array([7.0], f32)}
    c = O.lamb_ratio(np.array([3.0], f32), hp, ls)
    r = f32(1.0) + f32(0.1)
    _eq(ls["r_prev"], [r])
    _eq(c, [f32(2.0) * r])
    _eq(ls["c_prev"], c)
    _eq(ls["c_prev2"], [5.0])


# ---------------------------------------------------------------------------
# Warmup (uncompressed) steps
# ---------------------------------------------------------------------------

def test_warmup_adam_hand_two_workers():
    """[BLOG] §6 warmup with W = 2, by hand: g_bar = (g0 + g1)/2 = [4, 2];
    b1 = 0.5, b2 = 0.75: m = [2, 1], v = 0.25*g_bar^2 = [4, 1];
    u = m/(sqrt(v) + 0) = [1, 1]; p = -lr*u with lr = 0.25.  (u alone would
    not show a missing average: Adam's step is scale-free; m and v do.)"""
    lay = O.Layout(2, 2, 1, 1)
    g0 = np.array([2.0, 4.0], f32)
    g1 = np.array([6.0, 0.0], f32)
    m = np.zeros(lay.n_pad, f32)
    v = np.zeros(lay.n_pad, f32)
    p = np.zeros(lay.n_pad, f32)
    z = np.zeros(lay.n_pad - 2, f32)
    O.warmup_step(lay, [np.concatenate([g0, z]), np.concatenate([g1, z])], 0,
                  dict(b1=0.5, b2=0.75, eps=0.0, lr=0.25), m, v, p)
    _eq(m[:2], [2.0, 1.0])
    _eq(v[:2], [4.0, 1.0])
    _eq(p[:2], [-0.25, -0.25])


def test_warmup_adam_matches_torch_adam():
    """Warmup Adam has no bias correction.  torch.optim.Adam always corrects,
    so its lr and eps are rescaled per step to undo the correction:
    lr_t = lr * (1-b1^t) / sqrt(1-b2^t), eps_t = eps / sqrt(1-b2^t).
    One worker, so that the gradient average is exact on both sides (the
    average itself is pinned by the worked examples and by I5)."""
    torch = pytest.importorskip("torch")
    n, W = 3000, 1
    lay = O.Layout(n, W, 32, 1 << 20)
    rng = np.random.default_rng(21)
    hp = dict(b1=0.9, b2=0.999, eps=1e-8, lr=1e-3)
    m, v, p = (np.zeros(lay.n_pad, f32) for _ in range(3))
    p[:n] = rng.standard_normal(n).astype(f32) * f32(0.02)
    tp = torch.nn.Parameter(torch.tensor(p[:n].astype(np.float64)))
    # the oracle works in fp32: give torch the same (fp32-rounded) betas
    b1, b2 = float(f32(0.9)), float(f32(0.999))
    opt = torch.optim.Adam([tp], lr=hp["lr"], betas=(b1, b2), eps=hp["eps"])
    for t in range(1, 8):
        g = [np.zeros(lay.n_pad, f32) for _ in range(W)]
        for w in range(W):
            g[w][:n] = rng.standard_normal(n).astype(f32) * f32(1e-3)
        O.warmup_step(lay, g, 0, hp, m, v, p)
        bc1, bc2 = 1 - b1 ** t, 1 - b2 ** t
        for grp in opt.param_groups:
            grp["lr"] = hp["lr"] * bc1 / math.sqrt(bc2)
            grp["eps"] = hp["eps"] / math.sqrt(bc2)
        tp.grad = torch.tensor(np.mean([x[:n].astype(np.float64) for x in g], axis=0))
        opt.step()
        # fp32 vs fp64: a few units of rounding in each of about 10 operations
        # of every step (|u| <= 1/sqrt(1-b2) ~ 31.6), plus p's own rounding
        ref = tp.detach().numpy()
        tol = t * 10 * 2.0 ** -24 * hp["lr"] * 32 + np.spacing(np.abs(ref).astype(f32))
        assert np.all(np.abs(p[:n] - ref) <= tol)


def test_warmup_lamb_trust_ratio_hand():
    """One LAMB warmup step from m = v = 0 with b1 = 0.5, b2 = 0.75, eps = 0:
    m = 0.5 g, v = 0.25 g^2, u = m/sqrt(v) = sign(g).  Layer 0 has p = [3,4,0,0]
    (||p|| = 5) and ||u|| = 2, so c = 2.5 and p -= lr*2.5*u.  Layer 1 has
    p = 0, so c = 1."""
    lay = O.Layout(8, 1, 1, 8)
    layers = O.Layers([0, 4, 8])
    g = np.array([1, -2, 3, -4, 5, 6, -7, 8], f32)
    m, v = np.zeros(8, f32), np.zeros(8, f32)
    p = np.array([3, 4, 0, 0, 0, 0, 0, 0], f32)
    c_sum = np.zeros(2, f32)
    hp = dict(b1=0.5, b2=0.75, eps=0.0, lr=0.5, c_min=0.01, c_max=10.0)
    c = O.warmup_step(lay, [g], 1, hp, m, v, p, layers, c_sum)
    _eq(c, [2.5, 1.0])
    _eq(c_sum, [2.5, 1.0])
    _eq(m, 0.5 * g)
    _eq(v, 0.25 * g * g)
    _eq(p, [3 - 1.25, 4 + 1.25, -1.25, 1.25, -0.5, -0.5, 0.5, -0.5])


def test_lamb_begin_hand():
    """rms of layer 0 (m = 1,1,1,1) is 1, of layer 1 (m = 3,3,3,3) is 3; the
    mean is 2, so s = [2, 2/3]; c_avg = c_sum / T_w."""
    lay = O.Layout(8, 1, 1, 8)
    layers = O.Layers([0, 4, 8])
    m = np.array([1, 1, 1, 1, 3, 3, 3, 3], f32)
    ls = O.lamb_begin(lay, layers, m, np.array([3.0, 4.5], f32), 3)
    _eq(ls["s"], [2.0, f32(2.0) / f32(3.0)])
    _eq(ls["c_avg"], [1.0, 1.5])
    _eq(ls["c_prev"], [1.0, 1.5])
    _eq(ls["c_prev2"], [1.0, 1.5])
    _eq(ls["r_prev"], [1.0, 1.0])


# ---------------------------------------------------------------------------
# Philox4x32-10 and the INT8 stochastic-rounding quantizer
# ---------------------------------------------------------------------------

def _curand():
    cands = ["/usr/local/cuda/lib64/libcurand.so"] + sorted(
        glob.glob("/usr/local/cuda*/targets/*/lib/libcurand.so*"))
    for c in cands:
        try:
            return ct.CDLL(c)
        except OSError:
            continue
    pytest.skip("libcurand not found")


@pytest.mark.parametrize("seed", [0, 1234, 0x0123456789ABCDEF, 2 ** 64 - 1])
def test_philox_matches_curand_host_generator(seed):
    """curand's host Philox4x32-10 generator (run, not read) emits group i
    of 4 words from counter (i >> 16, 0, i & 0xffff, 0) under key = seed;
    the oracle's Philox must give the same words."""
    cr = _curand()
    gen = ct.c_void_p()
    assert cr.curandCreateGeneratorHost(ct.byref(gen), 161) == 0
    try:
        assert cr.curandSetPseudoRandomGeneratorSeed(gen, ct.c_ulonglong(seed)) == 0
        N = 1 << 20
        out = np.zeros(N, np.uint32)
        assert cr.curandGenerate(gen, out.ctypes.data_as(ct.c_void_p), ct.c_size_t(N)) == 0
    finally:
        cr.curandDestroyGenerator(gen)
    key = np.array([seed & 0xFFFFFFFF, seed >> 32], np.uint32)
    for i in [0, 1, 2, 3, 1000, 65535, 65536, 65537, 131071, 200000, 262143]:
        ctr = np.array([i >> 16, 0, i & 0xFFFF, 0], np.uint32)
        assert np.array_equal(O.philox4x32_10(ctr, key), out[4 * i: 4 * i + 4]), i


def test_uniform_uses_offset_and_subsequence_words():
    seed, step = 0xDEADBEEF12345678, 7
    key = np.array([seed & 0xFFFFFFFF, seed >> 32], np.uint32)
    for k in (0, 1, 2, 3, 4, 4097, (1 << 32) * 4 + 5):
        grp = k >> 2
        w = O.philox4x32_10(np.array([grp & 0xFFFFFFFF, grp >> 32, step, 0], np.uint32), key)
        assert O.uniform(seed, step, k) == f32(int(w[k & 3]) >> 8) / f32(1 << 24)


def test_uniform_is_uniform():
    u = np.array([O.uniform(1234, 3, k) for k in range(40000)], np.float64)
    assert np.all((u >= 0) & (u < 1))
    assert abs(u.mean() - 0.5) < 4 * math.sqrt(1 / 12 / u.size)
    hist = np.histogram(u, bins=10, range=(0, 1))[0]
    exp = u.size / 10
    chi2 = ((hist - exp) ** 2 / exp).sum()
    assert chi2 < 40  # 9 degrees of freedom; p < 1e-5 above this


def test_int8_block_pin_probabilities():
    """Block [127, -3.25, 0.5, 0, ...] has scale 127/127 = 1: 127 always codes
    as 127; -3.25 codes as -3 with probability 0.75 and -4 with 0.25; 0.5 as 0
    or 1 with 0.5 each; 0 as 0 (the tutorial's floor + Bernoulli(frac))."""
    g = np.zeros(256, f32)
    g[0], g[1], g[2] = 127.0, -3.25, 0.5
    N = 4000
    c1, c2 = 0, 0
    for step in range(N):
        q, sc = O.quant_int8(g, 256, seed=99, step=step)
        assert sc[0] == 1.0 and q[0] == 127 and np.all(q[3:] == 0)
        assert q[1] in (-3, -4) and q[2] in (0, 1)
        c1 += q[1] == -3
        c2 += q[2] == 1
    sd = math.sqrt(N * 0.25 * 0.75)
    assert abs(c1 - 0.75 * N) < 4 * sd
    assert abs(c2 - 0.5 * N) < 4 * math.sqrt(N * 0.25)


def test_int8_decision_follows_uniform():
    g = np.array([127.0, -3.25, 0.5, 2.75], f32)
    for step in range(50):
        q, _ = O.quant_int8(g, 4, seed=5, step=step)
        u = [O.uniform(5, step, k) for k in range(4)]
        assert q[1] == (-3 if u[1] < 0.75 else -4)
        assert q[2] == (1 if u[2] < 0.5 else 0)
        assert q[3] == (3 if u[3] < 0.75 else 2)


def test_int8_unbiased_over_seeds():
    """I7: E[q*scale] = g (the tutorial: stochastic rounding keeps the
    expectation)."""
    rng = np.random.default_rng(8)
    g = (rng.standard_normal(512) * 1e-3).astype(f32)
    N = 3000
    acc = np.zeros(512)
    for s in range(N):
        q, sc, d = O.quant_int8(g, 256, seed=1000 + s, step=0, deq=True)
        acc += d
    mean = acc / N
    scale = np.repeat(np.abs(g).reshape(2, 256).max(axis=1) / 127, 256)
    sd = 0.5 * scale / math.sqrt(N)   # the code is floor or floor+1
    assert np.all(np.abs(mean - g) < 4.5 * sd + 1e-12)


def test_int8_tie_rounds_down():
    """[TUT] "FP32 → INT8 量化" / GradientQuantizeINT8: q = floor(x) plus 1
    when the uniform is below the fraction, strictly.  A value whose
    fraction equals its own uniform exactly (scale 1: the block holds 127)
    rounds down; a comparison u <= frac would round it up."""
    seed, step = 77, 5
    u1 = O.uniform(seed, step, 1)
    q, sc = O.quant_int8(np.array([127.0, u1], f32), 256, seed=seed, step=step)
    assert sc[0] == f32(1.0)
    assert int(q[0]) == 127 and int(q[1]) == 0


def test_int8_code_clamped_to_127():
    """[TUT] GradientQuantizeINT8 clamps the code to +-127: the block's
    maximum can land just above 127 after x = g / (max/127) is rounded
    (max = 1.0000035 gives x = 127 + 2^-17), and when its uniform falls
    below that fraction the rounded-up 128 must be clamped back to 127.
    The element index is searched so that its uniform does fall below."""
    mx = f32(1.0)
    while True:  # the first float above 1 whose quotient exceeds 127
        mx = np.nextafter(mx, f32(2.0))
        x = mx / (mx / f32(127.0))
        if x > f32(127.0):
            break
    frac = x - np.floor(x)
    seed, step = 4321, 9
    k = next(k for k in range(3_000_000) if O.uniform(seed, step, k) < frac)
    k0 = k // 256 * 256
    g = np.zeros(256, f32)
    g[k - k0] = mx
    q, sc = O.quant_int8(g, 256, seed=seed, step=step, k0=k0)
    assert sc[0] == mx / f32(127.0)
    assert int(q[k - k0]) == 127


def test_int8_edges():
    q, sc = O.quant_int8(np.zeros(300, f32), 256)
    assert np.all(q == 0) and np.all(sc == 0)
    rng = np.random.default_rng(1)
    g = (rng.standard_normal(1000) * 10).astype(f32)
    q, sc, d = O.quant_int8(g, 256, seed=3, step=1, deq=True)
    assert len(sc) == 4 and q.min() >= -127 and q.max() <= 127
    blocks = [g[i:i + 256] for i in range(0, 1000, 256)]
    for b, s in zip(blocks, sc):
        assert s == f32(np.abs(b).max()) / f32(127)
    _eq(d, q.astype(f32) * np.repeat(sc, 256)[:1000])


def test_int8_whole_tensor_equals_page_function():
    """With one block over the whole tensor the quantizer is the tutorial's
    GradientQuantizeINT8.backward, given the same uniforms r."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(2)
    g = (rng.standard_normal(777) * 1e-2).astype(f32)
    q, sc, d = O.quant_int8(g, 777, seed=42, step=9, deq=True)
    r = torch.tensor([O.uniform(42, 9, k) for k in range(777)])
    go = torch.tensor(g)
    max_val = torch.max(torch.abs(go))
    scale = max_val / 127
    gs = go / scale
    gi = torch.floor(gs)
    gi += (r < (gs - gi)).float()
    qq = torch.clamp(gi, -127, 127)
    assert np.array_equal(qq.numpy().astype(np.int8), q)
    assert np.array_equal((qq * scale).numpy(), d)


# ---------------------------------------------------------------------------
# Stability variants of the "1bit Adam" write-up, 4.1
# ---------------------------------------------------------------------------

def test_clip_of_the_compensated_value_hand():
    """b1 = 0 and e = 0 make x = g; clip 2 turns [3, -5, 1, 0.5] into
    [2, -2, 1, 0.5]: scale (2+2+1+0.5)/4 = 1.375, e' = x - 1.375*sign(x)."""
    lay = O.Layout(4, 1, 1, 4)
    g = np.array([3.0, -5.0, 1.0, 0.5], f32)
    e = np.zeros(4, f32)
    b, s, x = O.compress_worker(lay, g, np.zeros(4, f32), e, 0.0, clip=2.0)
    _eq(x, [2.0, -2.0, 1.0, 0.5])
    _eq(s, [1.375])
    _eq(e, [0.625, -0.625, -0.375, -0.875])
    assert int(b[0]) == 0b1101
    # a NaN stays NaN under the clamp
    g[1] = np.nan
    b, s, x = O.compress_worker(lay, g, np.zeros(4, f32), np.zeros(4, f32), 0.0, clip=2.0)
    assert np.isnan(x[1]) and not (int(b[0]) >> 1) & 1


def test_clip_zero_is_off():
    lay, g, m, e = _rand_case()
    e1, e2 = e[0].copy(), e[0].copy()
    b1_, s1, x1 = O.compress_worker(lay, g[0], m, e1, 0.9)
    b2_, s2, x2 = O.compress_worker(lay, g[0], m, e2, 0.9, clip=0.0)
    _eq(x1, x2)
    _eq(e1, e2)


def test_reset_then_step_equals_fresh_start():
    """After the periodic reset the next step sees e = 0, e_s = 0: it equals
    a step from a state whose errors were never set."""
    lay = O.Layout(3000, 2, 32, 512)
    rng = np.random.default_rng(31)
    hp = dict(b1=0.9, b2=0.999, eps=1e-8, lr=1e-4)
    a = O.State(lay)
    a.v[:3000] = np.abs(rng.standard_normal(3000)).astype(f32) * f32(1e-6) + f32(1e-8)
    g = [np.zeros(lay.n_pad, f32) for _ in range(2)]
    for w in range(2):
        g[w][:3000] = rng.standard_normal(3000).astype(f32) * f32(1e-3)
    O.compressed_step(a, g, hp)
    b = a.copy()
    O.reset_errors(a)
    for e in b.e:
        e[:] = 0
    b.e_s[:] = 0
    O.compressed_step(a, g, hp)
    O.compressed_step(b, g, hp)
    _eq(a.p, b.p)
    assert all(np.array_equal(x, y) for x, y in zip(a.e, b.e))


# ---------------------------------------------------------------------------
# INT8 with error feedback and the error monitor
# ---------------------------------------------------------------------------

def test_int8_ef_zero_error_is_plain_int8():
    """With e = 0 the codes and scales are those of the plain quantizer, and
    the residual is x - q*scale."""
    rng = np.random.default_rng(40)
    g = (rng.standard_normal(1000) * 1e-3).astype(f32)
    e = np.zeros(1000, f32)
    q, sc, d = O.quant_int8_ef(g, e, seed=3, step=4, deq=True)
    q0, sc0, d0 = O.quant_int8(g, 256, 3, 4, deq=True)
    assert np.array_equal(q, q0)
    _eq(sc, sc0)
    _eq(e, (g - d0).astype(f32))


def test_int8_ef_hand_block():
    """x = g + e = [254, -7, 1, 0.25 ...]: scale 2; x/scale = [127, -3.5, 0.5,
    0.125]; codes 127 always, -3 or -4, 0 or 1, 0 or 1; residual x - q*2."""
    g = np.zeros(256, f32)
    e = np.zeros(256, f32)
    g[:4] = [250.0, -7.0, 1.0, 0.0]
    e[:4] = [4.0, 0.0, 0.0, 0.25]
    q, sc, d, e2 = O.quant_int8_ef(g, e, seed=11, step=0, deq=True, err2=True)
    assert sc[0] == 2.0 and q[0] == 127 and e[0] == 0.0
    assert q[1] in (-3, -4) and e[1] == -7.0 - 2.0 * q[1]
    assert q[2] in (0, 1) and e[2] == 1.0 - 2.0 * q[2]
    assert q[3] in (0, 1) and e[3] == 0.25 - 2.0 * q[3]
    # the monitor: one value per block, the sum of the squared residuals
    assert e2[0] == f32(e[1] ** 2 + e[2] ** 2 + e[3] ** 2)


def test_int8_ef_residual_stays_bounded_and_unbiased():
    """Error feedback keeps |e| within one quantisation step, and the
    dequantised sum tracks the true sum (the telescoping of the write-up's
    2.1 claim, E[sum q] = E[sum g])."""
    rng = np.random.default_rng(41)
    g = (rng.standard_normal(512) * 1e-3).astype(f32)
    e = np.zeros(512, f32)
    total_q = np.zeros(512)
    for t in range(200):
        q, sc, d = O.quant_int8_ef(g, e, seed=1, step=t, deq=True)
        total_q += d
        step = np.repeat(sc, 256)
        assert np.all(np.abs(e) <= step * (1 + 1e-6) + 1e-12)
    # sum of the dequantised values = sum of g minus the final residual
    assert np.allclose(total_q, 200 * g.astype(np.float64) - e, rtol=0, atol=1e-6)
