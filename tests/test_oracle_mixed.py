"""Pins for the oracle's layerwise mixed-width codecs (the b-bit block
quantizer with error feedback and the FP16 codec sent every 10th step, as
read from the "1bit Adam" write-up's §3.2 table and §6 layerwise_bits, and
from the quantizer of "梯度量化：将梯度从 FP32 压到 INT8 甚至 1-bit").

Each test checks oracle/ against something other than itself: NumPy's
binary16 conversion, the tutorial's GradientQuantizeINT8 function (which
takes the width as an argument) run in torch, the oracle's independently
pinned INT8 quantizer, hand-computed values, statistics and the
error-feedback identity.  No GPU is needed.
"""
import math

import numpy as np
import pytest

import oracle as O

f32 = np.float32


def _eq(a, b):
    a = np.asarray(a, np.float32)
    b = np.asarray(b, np.float32)
    assert a.shape == b.shape
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), (a, b)


def _unpack(codes, bits, count):
    """Two's-complement fields of `bits` bits, LSB first (test-side reading
    of the documented layout)."""
    out = np.zeros(count, np.int64)
    for k in range(count):
        bit = k * bits
        f = (int(codes[bit // 32]) >> (bit % 32)) & ((1 << bits) - 1)
        out[k] = f - (1 << bits) if f >= (1 << (bits - 1)) else f
    return out


# ---------------------------------------------------------------------------
# binary16 conversion
# ---------------------------------------------------------------------------

def test_f16_decode_all_patterns_matches_numpy():
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = O.f16_to_f32(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_f16_encode_matches_numpy():
    """Round trip of every finite half, every midpoint between neighbours
    (the ties, which go to the even neighbour), one float32 ulp either side
    of each midpoint, the overflow edge and random values over 47 binades."""
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = h.view(np.float16).astype(np.float64)
    fin = np.isfinite(v)
    pos = np.sort(np.unique(v[fin & (v >= 0)]))
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)       # exact in float32
    assert np.array_equal(mids.astype(np.float64), (pos[:-1] + pos[1:]) / 2)
    up = np.nextafter(mids, np.float32(np.inf))
    dn = np.nextafter(mids, np.float32(0))
    rng = np.random.default_rng(4)
    rnd = (2.0 ** rng.uniform(-30, 17, 60000)).astype(f32)
    edge = np.array([65504, 65519.996, 65520, 65536, 1e9, np.inf, 0.0,
                     2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -24, 2.0 ** -14,
                     2.0 ** -14 - 2.0 ** -25], f32)
    xs = np.concatenate([v[fin].astype(f32), mids, up, dn, rnd, edge])
    xs = np.concatenate([xs, -xs])
    ours = O.f32_to_f16(xs)
    with np.errstate(over="ignore"):
        ref = xs.astype(np.float16).view(np.uint16)
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, [(float(xs[i]), hex(ours[i]), hex(ref[i])) for i in bad[:5]]


def test_f16_nan_is_quiet_nan():
    h = O.f32_to_f16(np.array([np.nan, -np.nan], f32))
    assert np.all(np.isnan(h.view(np.float16)))


# ---------------------------------------------------------------------------
# The b-bit block quantizer
# ---------------------------------------------------------------------------

def _one_worker(bits, g, seed, step, n=None, e=None):
    """Worker 0 of W = 1 with b1 = 0 and m = 0, so x = g + e."""
    n = g.size if n is None else n
    lay = O.Layout(n, 1, 256, 256)
    gp = np.zeros(lay.n_pad, f32)
    gp[:g.size] = g
    ep = np.zeros(lay.n_pad, f32) if e is None else e
    codes, sc = O.qb_compress_worker(lay, bits, gp, np.zeros(lay.n_pad, f32), ep, 0.0, 0,
                                     seed, step)
    return lay, codes, sc, ep


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_qb_one_block_equals_page_function(bits):
    """One block of 256 is the tutorial's GradientQuantizeINT8.backward with
    its `bits` argument, given the same uniforms r (run in torch)."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(bits)
    g = (rng.standard_normal(256) * 1e-2).astype(f32)
    seed, step = 77, 3
    lay, codes, sc, e = _one_worker(bits, g, seed, step)
    r = torch.tensor([O.uniform(seed, step, k) for k in range(256)])
    go = torch.tensor(g)
    max_val = torch.max(torch.abs(go))
    scale = max_val / (2 ** (bits - 1) - 1)
    gs = go / scale
    gi = torch.floor(gs)
    gi += (r < (gs - gi)).float()
    q = torch.clamp(gi, -2 ** (bits - 1) + 1, 2 ** (bits - 1) - 1)
    assert np.array_equal(_unpack(codes, bits, 256), q.numpy().astype(np.int64))
    _eq(sc[0], scale.numpy())
    _eq(g - O.qb_decode(lay, bits, codes, sc), e)   # e' = x - q*scale


def test_qb8_equals_int8_with_error_feedback():
    """Width 8 with b1 = 0 (x = g + e) is the INT8 quantizer with error
    feedback, whose uniforms are counted from w*n_pad for worker w; the
    server of W = 1 is the same quantizer applied to e_s + q*scale with the
    uniforms counted from n_pad."""
    n, W = 3000, 3
    lay = O.Layout(n, W, 256, 256)
    rng = np.random.default_rng(5)
    for w in range(W):
        g = np.zeros(lay.n_pad, f32)
        g[:n] = rng.standard_normal(n).astype(f32) * f32(1e-3)
        e1 = np.zeros(lay.n_pad, f32)
        e1[:n] = rng.standard_normal(n).astype(f32) * f32(1e-4)
        e2 = e1.copy()
        codes, sc = O.qb_compress_worker(lay, 8, g, np.zeros(lay.n_pad, f32), e1, 0.0, w,
                                         seed=9, step=4)
        q, sc2 = O.quant_int8_ef(g, e2, seed=9, step=4, k0=w * lay.n_pad)
        assert np.array_equal(codes.view(np.int8), q)
        _eq(sc, sc2)
        _eq(e1, e2)
    lay1 = O.Layout(n, 1, 256, 256)
    g = np.zeros(lay1.n_pad, f32)
    g[:n] = rng.standard_normal(n).astype(f32) * f32(1e-3)
    e = np.zeros(lay1.n_pad, f32)
    codes, sc = O.qb_compress_worker(lay1, 8, g, np.zeros_like(g), e, 0.0, 0, 9, 4)
    e_s = np.zeros(lay1.n_pad, f32)
    e_s[:n] = rng.standard_normal(n).astype(f32) * f32(1e-4)
    e_s2 = e_s.copy()
    sco, ssc = O.qb_server(lay1, 8, codes[None], sc[None], e_s, 9, 4)
    z = O.qb_decode(lay1, 8, codes, sc)
    q, ss2 = O.quant_int8_ef(z, e_s2, seed=9, step=4, k0=lay1.n_pad)
    assert np.array_equal(sco.view(np.int8), q)
    _eq(ssc, ss2)
    _eq(e_s, e_s2)


def test_qb2_hand_block():
    """Block [2, -1, 0.5, 0, ...]: scale = 2/1 = 2; 2 codes as 1 (error 0);
    -1 is -0.5 scales: -1 or 0 with probability 1/2 each (error +1 or -1);
    0.5 is 0.25 scales: 1 with probability 1/4 (error -1.5), else 0 (error
    0.5); fields of 2 bits, LSB first, -1 as 0b11."""
    g = np.zeros(256, f32)
    g[:3] = [2.0, -1.0, 0.5]
    N = 4000
    c1 = c2 = 0
    for step in range(N):
        lay, codes, sc, e = _one_worker(2, g, seed=21, step=step)
        q = _unpack(codes, 2, 256)
        assert sc[0] == 2.0 and q[0] == 1 and np.all(q[3:] == 0)
        assert e[0] == 0.0 and np.all(e[3:] == 0.0)
        u1, u2 = O.uniform(21, step, 1), O.uniform(21, step, 2)
        assert q[1] == (0 if u1 < 0.5 else -1)
        assert q[2] == (1 if u2 < 0.25 else 0)
        assert e[1] == (-1.0 if q[1] == 0 else 1.0)
        assert e[2] == (-1.5 if q[2] == 1 else 0.5)
        w0 = 1 | ((q[1] & 3) << 2) | ((q[2] & 3) << 4)
        assert int(codes[0]) == w0 and np.all(codes[1:] == 0)
        c1 += q[1] == 0
        c2 += q[2] == 1
    assert abs(c1 - N / 2) < 4 * math.sqrt(N / 4)
    assert abs(c2 - N / 4) < 4 * math.sqrt(N * 3 / 16)


@pytest.mark.parametrize("bits", [2, 4])
def test_qb_unbiased(bits):
    """E[q*scale] = x: stochastic rounding keeps the expectation (the
    tutorial's reason for it)."""
    rng = np.random.default_rng(10 + bits)
    g = (rng.standard_normal(512) * 1e-3).astype(f32)
    N = 2000
    acc = np.zeros(512)
    for s in range(N):
        lay, codes, sc, _ = _one_worker(bits, g, seed=500, step=s)
        acc += O.qb_decode(lay, bits, codes, sc)
    mean = acc / N
    scale = np.repeat(np.abs(g).reshape(2, 256).max(axis=1) / (2 ** (bits - 1) - 1), 256)
    sd = 0.5 * scale / math.sqrt(N)
    assert np.all(np.abs(mean - g) < 4.5 * sd + 1e-12)


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_qb_codes_in_range_and_error_identity(bits):
    """Codes lie in [-(2^(b-1)-1), 2^(b-1)-1] and are the floor or floor+1 of
    x/scale; x = q*scale + e' within an ulp; padding codes 0 with error 0."""
    n = 1000
    rng = np.random.default_rng(3)
    g = (rng.standard_normal(n) * 10.0 ** rng.uniform(-4, 0, n)).astype(f32)
    lay, codes, sc, e = _one_worker(bits, g, seed=1, step=2, n=n)
    q = _unpack(codes, bits, lay.n_pad)
    qmax = 2 ** (bits - 1) - 1
    assert q.min() >= -qmax and q.max() <= qmax
    assert np.all(q[n:] == 0) and np.all(e[n:] == 0)
    s = np.repeat(sc, 256)[:n].astype(np.float64)
    xs = g.astype(np.float64) / s
    assert np.all((q[:n] == np.floor(xs)) | (q[:n] == np.floor(xs) + 1) |
                  (np.abs(xs) >= qmax))
    back = q[:n] * s + e[:n]
    tol = 2.0 ** -23 * np.maximum(np.abs(g), np.abs(e[:n]))
    assert np.all(np.abs(back - g) <= tol)
    for b in range(4):
        blk = g[256 * b: 256 * (b + 1)]
        assert sc[b] == f32(np.abs(blk).max()) / f32(qmax)


def test_qb_lower_clamp():
    """x/scale can fall just below -(2^(b-1)-1) through the rounding of
    max/(2^(b-1)-1): for b = 4 and x = -v, v = 1 + 6*2^-23, x/scale is
    -7.0000005 (floor -8, frac 1 - 2^-21).  With a uniform above that frac
    the unclamped code would be -8; the clamp makes it -7.  (seed 1234, step
    266379 were found by scanning steps for such a uniform at element 0.)"""
    v = f32(1) + f32(6) * f32(2.0 ** -23)
    s = v / f32(7)
    xs = -v / s
    assert xs < f32(-7)
    frac = xs - np.floor(xs)
    assert O.uniform(1234, 266379, 0) >= frac
    g = np.zeros(256, f32)
    g[0], g[1] = -v, f32(0.5)
    lay, codes, sc, e = _one_worker(4, g, seed=1234, step=266379)
    q = _unpack(codes, 4, 256)
    assert sc[0] == s and q[0] == -7
    _eq(e[0], -v - f32(-7) * s)


def test_qb_zero_block_and_nan():
    g = np.zeros(512, f32)
    g[300] = np.nan
    g[301] = 1.0
    lay, codes, sc, e = _one_worker(2, g, seed=1, step=1)
    q = _unpack(codes, 2, 512)
    assert sc[0] == 0.0 and np.all(q[:256] == 0)
    assert sc[1] == 1.0 and q[300 - 0] == 0 and q[301] == 1


def test_qb_adam_hand():
    """m = q*scale = 1*0.5; p = 1 - 0.125*(0.5/(sqrt(4)+0)) = 0.96875."""
    lay = O.Layout(256, 1, 256, 256)
    codes = np.zeros(O.qb_words(256, 2), np.uint32)
    codes[0] = 1                      # element 0: q = 1
    codes[0] |= 3 << 2                # element 1: q = -1
    sc = np.array([0.5], f32)
    v = np.full(256, 4.0, f32)
    m = np.zeros(256, f32)
    p = np.ones(256, f32)
    O.qb_adam(lay, 2, codes, sc, v, 0.0, 0.125, m, p)
    assert m[0] == 0.5 and m[1] == -0.5 and np.all(m[2:] == 0)
    assert p[0] == 0.96875 and p[1] == 1.03125 and np.all(p[2:] == 1.0)


# ---------------------------------------------------------------------------
# FP16 codec
# ---------------------------------------------------------------------------

def test_f16_codec_hand_example():
    """W = 2, b1 = 0: x0 = 1 + 2^-11 is a tie and rounds to 1 (error 2^-11);
    x1 = 1 + 3*2^-11 is a tie and rounds to the even 1 + 2^-9 (error
    -2^-11); the server's average 1 + 2^-10 is exact (e_s 0); with v = 4,
    eps = 0, lr = 0.5 the parameter moves by (1 + 2^-10)/4."""
    lay = O.Layout(32, 2, 32, 32)
    assert lay.P == 32 and lay.n_pad == 64
    g = [np.zeros(64, f32), np.zeros(64, f32)]
    g[0][0] = 1 + 2.0 ** -11
    g[1][0] = 1 + 3 * 2.0 ** -11
    e = [np.zeros(64, f32), np.zeros(64, f32)]
    h = np.zeros((2, 64), np.uint16)
    m = np.zeros(64, f32)
    for w in range(2):
        O.f16_compress_worker(lay, g[w], m, e[w], 0.0, True, h[w])
    assert O.f16_to_f32(h[0, :1])[0] == 1.0 and e[0][0] == 2.0 ** -11
    assert O.f16_to_f32(h[1, :1])[0] == 1 + 2.0 ** -9 and e[1][0] == -2.0 ** -11
    e_s = np.zeros(64, f32)
    hs = O.f16_server(lay, h, e_s)
    assert O.f16_to_f32(hs[:1])[0] == 1 + 2.0 ** -10 and np.all(e_s == 0)
    v = np.full(64, 4.0, f32)
    p = np.full(64, 3.0, f32)
    O.f16_adam(lay, True, hs, v, 0.0, 0.5, m, p)
    assert m[0] == 1 + 2.0 ** -10 and p[0] == 3.0 - (1 + 2.0 ** -10) / 4
    assert np.all(p[1:] == 3.0)


def test_f16_non_sending_step_keeps_everything():
    """Off the 10th steps nothing is sent: e' = x exactly, m = 0, p, h and
    e_s untouched."""
    lay = O.Layout(100, 2, 32, 32)
    rng = np.random.default_rng(0)
    g = rng.standard_normal(lay.n_pad).astype(f32)
    g[100:] = 0
    m = rng.standard_normal(lay.n_pad).astype(f32)
    m[100:] = 0
    e = rng.standard_normal(lay.n_pad).astype(f32)
    e[100:] = 0
    e0 = e.copy()
    h = np.full(lay.n_pad, 7, np.uint16)
    O.f16_compress_worker(lay, g, m, e, 0.9, False, h)
    assert np.all(h == 7)
    # x = (0.9*m + 0.1*g) + e, each operation rounded in float32
    x = (f32(0.9) * m + (f32(1) - f32(0.9)) * g) + e0
    _eq(e[:100], x[:100])
    p = rng.standard_normal(lay.n_pad).astype(f32)
    p0 = p.copy()
    O.f16_adam(lay, False, np.zeros(lay.n_pad, np.uint16), np.ones(lay.n_pad, f32), 1e-8,
               1e-3, m, p)
    assert np.all(m == 0)
    _eq(p, p0)


# ---------------------------------------------------------------------------
# The error-feedback identity over whole steps
# ---------------------------------------------------------------------------

def _delta(st):
    return np.mean([e.astype(np.float64) for e in st.e], axis=0) + st.e_s


@pytest.mark.parametrize("bits", [2, 4, 16])
def test_i5_identity_mixed_codecs(bits):
    """m_t = b1*m_{t-1} + (1-b1)*g_bar + delta~_{t-1} - delta~_t with
    delta~ = mean_w e_w + e_s (the 1-bit LAMB summary's global-momentum
    identity), on every step of every codec, sending or not."""
    n, W = 3000, 3
    lay = O.Layout(n, W, 256, 1024)
    st = O.State(lay)
    rng = np.random.default_rng(bits)
    st.v[:n] = np.abs(rng.standard_normal(n)).astype(f32) * f32(1e-6) + f32(1e-8)
    st.m[:n] = rng.standard_normal(n).astype(f32) * f32(1e-3)
    hp = dict(b1=0.9, b2=0.999, eps=1e-8, lr=1e-4)
    d_prev = _delta(st)
    for t in range(1, 8):
        g = [np.zeros(lay.n_pad, f32) for _ in range(W)]
        for w in range(W):
            g[w][:n] = rng.standard_normal(n).astype(f32) * f32(1e-3)
        gbar = np.mean([x.astype(np.float64) for x in g], axis=0)
        m_prev = st.m.astype(np.float64)
        O.codec_step(st, g, hp, bits, t, seed=3, period=3)
        d = _delta(st)
        rhs = 0.9 * m_prev + 0.1 * gbar + d_prev - d
        scale = np.abs(m_prev).max() + np.abs(d).max() + np.abs(gbar).max()
        assert np.max(np.abs(st.m[:n] - rhs[:n])) <= 64 * 2.0 ** -24 * scale
        if bits == 16 and t % 3:
            assert np.all(st.m == 0)
        assert np.all(st.m[n:] == 0)
        assert all(np.all(e[n:] == 0) for e in st.e) and np.all(st.e_s[n:] == 0)
        d_prev = d


def test_codec_step_width_one_is_the_scaled_sign_step():
    n, W = 2000, 2
    lay = O.Layout(n, W, 256, 512)
    a, b = O.State(lay), O.State(lay)
    rng = np.random.default_rng(1)
    v = np.abs(rng.standard_normal(lay.n_pad)).astype(f32) + f32(1e-3)
    a.v[:] = v
    b.v[:] = v
    g = [rng.standard_normal(lay.n_pad).astype(f32) for _ in range(W)]
    for x in g:
        x[n:] = 0
    hp = dict(b1=0.9, b2=0.999, eps=1e-8, lr=1e-4)
    O.codec_step(a, g, hp, 1, 1, seed=0)
    O.compressed_step(b, g, hp)
    _eq(a.p, b.p)
    _eq(a.m, b.m)
