"""Python face of the oracle (oracle/oracle.cpp) over NumPy arrays.

TEST INFRASTRUCTURE ONLY: tests/, __graft_entry__.smoke() and the CPU
baseline leg of bench.py may import this package; the product path
(momentum_compression_gb300) never does.  Every function here marshals
arguments and calls the C oracle; the arithmetic lives in oracle.cpp, where
each function cites the passage it follows.
"""
import ctypes as ct
import os

import numpy as np

from . import build as _build

_lib = None


class _Layout(ct.Structure):
    _fields_ = [(k, ct.c_uint64) for k in
                ("n", "W", "A", "C", "P", "n_pad", "cpp", "nc")]


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ct.CDLL(path)
        f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
        u32p = np.ctypeslib.ndpointer(np.uint32, flags="C_CONTIGUOUS")
        u64p = np.ctypeslib.ndpointer(np.uint64, flags="C_CONTIGUOUS")
        i8p = np.ctypeslib.ndpointer(np.int8, flags="C_CONTIGUOUS")
        vp = ct.c_void_p
        u64, f32 = ct.c_uint64, ct.c_float
        L.orc_make_layout.argtypes = [u64, u64, u64, u64, ct.POINTER(_Layout)]
        L.orc_make_layout.restype = ct.c_int
        L.orc_cr_sum.argtypes = [f32p, u64]
        L.orc_cr_sum.restype = f32
        lay = ct.POINTER(_Layout)
        L.orc_compress_worker.argtypes = [lay, vp, u64, vp, vp, f32, f32p, f32p,
                                          f32p, u32p, f32p, vp]
        L.orc_compress_worker_clip.argtypes = [lay, vp, u64, vp, vp, f32, f32, f32p, f32p,
                                               f32p, u32p, f32p, vp]
        L.orc_server_reduce.argtypes = [lay, vp, u64, vp, u32p, f32p, f32p,
                                        u32p, f32p, vp]
        L.orc_error_norm.argtypes = [lay, f32p, f32p]
        L.orc_compress_worker_range.argtypes = [lay, vp, u64, vp, vp, f32, f32, f32p, f32p,
                                                f32p, u32p, f32p, vp, u64, u64]
        L.orc_server_reduce_range.argtypes = [lay, vp, u64, vp, u32p, f32p, f32p, u32p, f32p,
                                              vp, u64, u64]
        L.orc_lamb_pass_a_range.argtypes = [lay, vp, u64, f32p, u32p, f32p, f32p, f32, f32,
                                            f32p, f32p, f32p, u64, u64]
        L.orc_lamb_pass_b_range.argtypes = [lay, vp, u64, f32p, f32p, f32p, f32, f32, f32p,
                                            u64, u64]
        L.orc_decompress.argtypes = [lay, vp, u64, vp, u32p, f32p, f32p]
        L.orc_adam_update.argtypes = [lay, u32p, f32p, f32p, f32, f32, f32p, f32p]
        L.orc_lamb_pass_a.argtypes = [lay, vp, u64, f32p, u32p, f32p, f32p, f32,
                                      f32, f32p, f32p, f32p]
        L.orc_lamb_ratio.argtypes = [u64, f32p, f32, f32, f32, f32, f32, ct.c_int,
                                     f32p, f32p, f32p, f32p, f32p]
        L.orc_lamb_rho.argtypes = [u64, f32p, f32p, f32p]
        L.orc_lamb_pass_b.argtypes = [lay, vp, u64, f32p, f32p, f32p, f32, f32,
                                      f32p]
        L.orc_warmup_step.argtypes = [lay, vp, u64, ct.POINTER(ct.c_void_p),
                                      ct.c_int, f32, f32, f32, f32, f32, f32,
                                      f32p, f32p, f32p, vp, vp]
        L.orc_lamb_begin.argtypes = [lay, vp, u64, f32p, f32p, u64, f32p, f32p,
                                     f32p, f32p, f32p]
        L.orc_philox4x32_10.argtypes = [u32p, u32p, u32p]
        L.orc_uniform.argtypes = [u64, u64, u64]
        L.orc_uniform.restype = f32
        L.orc_quant_int8.argtypes = [f32p, u64, u64, u64, u64, i8p, f32p,
                                     vp]
        L.orc_quant_int8_at.argtypes = [f32p, u64, u64, u64, u64, u64, i8p, f32p, vp]
        L.orc_quant_int8_ef_at.argtypes = [f32p, f32p, u64, u64, u64, u64, i8p, f32p, vp, vp]
        u16p = np.ctypeslib.ndpointer(np.uint16, flags="C_CONTIGUOUS")
        ci = ct.c_int
        L.orc_qb_compress_worker_at.argtypes = [lay, ci, f32, f32, u64, u64, u64, u64, u64,
                                                f32p, f32p, f32p, u32p, f32p]
        L.orc_qb_server_at.argtypes = [lay, ci, u64, u64, u64, u64, u32p, u64, f32p, u64,
                                       f32p, u32p, f32p]
        L.orc_qb_decode_at.argtypes = [lay, ci, u64, u64, u32p, f32p, f32p]
        L.orc_qb_adam_at.argtypes = [lay, ci, f32, f32, u64, u64, u32p, f32p, f32p, f32p,
                                     f32p]
        L.orc_f32_to_f16.argtypes = [f32]
        L.orc_f32_to_f16.restype = ct.c_uint16
        L.orc_f16_to_f32.argtypes = [ct.c_uint16]
        L.orc_f16_to_f32.restype = f32
        L.orc_f16_compress_worker.argtypes = [lay, f32, f32, ci, f32p, f32p, f32p, u16p]
        L.orc_f16_server.argtypes = [lay, u16p, f32p, u16p]
        L.orc_f16_adam.argtypes = [lay, ci, f32, f32, u16p, f32p, f32p, f32p]
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ct.c_void_p)


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


class Layout:
    """n, W, alignment A, chunk C -> P, n_pad, chunks per partition, chunks."""

    def __init__(self, n, W, A=4096, C=1 << 20):
        self._s = _Layout()
        if lib().orc_make_layout(n, W, A, C, ct.byref(self._s)) != 0:
            raise ValueError("invalid layout")
        for k, _ in _Layout._fields_:
            setattr(self, k, int(getattr(self._s, k)))
        self.words = (self.n_pad + 31) // 32

    def chunk_range(self, g):
        j, kc = divmod(g, self.cpp)
        s = j * self.P + kc * self.C
        ln = min(self.C, self.P - kc * self.C)
        real = max(0, min(self.n - s, ln))
        return s, ln, real


class Layers:
    """Per-layer offsets of the fused buffer (None = one layer)."""

    def __init__(self, offsets=None):
        if offsets is None:
            self.off, self.nl = None, 0
        else:
            self.off = np.ascontiguousarray(offsets, dtype=np.uint64)
            self.nl = len(self.off) - 1

    def count(self):
        return max(self.nl, 1)


def cr_sum(a):
    a = _f32(a)
    return np.float32(lib().orc_cr_sum(a, a.size))


def compress_worker(lay, g, m, e, b1, layers=None, sigma=None, rho=None, clip=0.0,
                    want_x=True):
    """One worker's compression.  e (n_pad,) is updated in place.  clip > 0
    limits the compensated value to [-clip, clip].
    Returns (bits[words] u32, scales[nc] f32, x[n_pad] f32); x is None when
    want_x is False (saves an n_pad array on whole-model sizes)."""
    layers = layers or Layers()
    bits = np.zeros(lay.words, np.uint32)
    scales = np.zeros(lay.nc, np.float32)
    x = np.zeros(lay.n_pad, np.float32) if want_x else None
    sg = None if sigma is None else _f32(sigma)
    rh = None if rho is None else _f32(rho)
    lib().orc_compress_worker_clip(lay._s, _ptr(layers.off), layers.nl, _ptr(sg),
                                   _ptr(rh), b1, clip, _f32(g), _f32(m), e, bits,
                                   scales, _ptr(x))
    return bits, scales, x


def server_reduce(lay, bits, scales, e_s, layers=None, rho=None, want_y=True):
    """bits (W, words) u32, scales (W, nc) f32; e_s (n_pad,) updated in place.
    Returns (sbits[words], sscales[nc], y[n_pad]); y is None when want_y is
    False."""
    layers = layers or Layers()
    bits = np.ascontiguousarray(bits, dtype=np.uint32)
    scales = _f32(scales)
    sbits = np.zeros(lay.words, np.uint32)
    sscales = np.zeros(lay.nc, np.float32)
    y = np.zeros(lay.n_pad, np.float32) if want_y else None
    rh = None if rho is None else _f32(rho)
    lib().orc_server_reduce(lay._s, _ptr(layers.off), layers.nl, _ptr(rh),
                            bits.reshape(-1), scales.reshape(-1), e_s, sbits,
                            sscales, _ptr(y))
    return sbits, sscales, y


# Chunk ranges: the same computations for chunks g0 <= g < g1 only, writing
# into the caller's whole-buffer arrays.  Disjoint ranges whose boundaries
# fall on multiples of 32 elements may run in concurrent threads (the C
# calls release the GIL); pass A returns the range's R, merged by maximum.

def compress_worker_range(lay, g0, g1, g, m, e, bits, scales, b1, layers=None, sigma=None,
                          rho=None, clip=0.0):
    """compress_worker over chunks [g0, g1): e, bits (words,) and scales
    (nc,) are updated in place for those chunks' elements."""
    layers = layers or Layers()
    sg = None if sigma is None else _f32(sigma)
    rh = None if rho is None else _f32(rho)
    lib().orc_compress_worker_range(lay._s, _ptr(layers.off), layers.nl, _ptr(sg), _ptr(rh),
                                    b1, clip, g, m, e, bits, scales, None, g0, g1)


def server_reduce_range(lay, g0, g1, bits, scales, e_s, sbits, sscales, layers=None, rho=None):
    """server_reduce over chunks [g0, g1): e_s, sbits and sscales updated in
    place for those chunks."""
    layers = layers or Layers()
    rh = None if rho is None else _f32(rho)
    lib().orc_server_reduce_range(lay._s, _ptr(layers.off), layers.nl, _ptr(rh),
                                  np.ascontiguousarray(bits, dtype=np.uint32).reshape(-1),
                                  _f32(scales).reshape(-1), e_s, sbits, sscales, None, g0, g1)


def lamb_pass_a_range(lay, g0, g1, layers, sigma, sbits, sscales, v_frozen, b1, b2, m,
                      v_fresh):
    """lamb_pass_a over chunks [g0, g1); returns that range's R."""
    R = np.zeros(layers.count(), np.float32)
    lib().orc_lamb_pass_a_range(lay._s, _ptr(layers.off), layers.nl, _f32(sigma),
                                np.ascontiguousarray(sbits, np.uint32), _f32(sscales),
                                _f32(v_frozen), b1, b2, m, v_fresh, R, g0, g1)
    return R


def lamb_pass_b_range(lay, g0, g1, layers, c, m, v_frozen, eps, lr, p):
    lib().orc_lamb_pass_b_range(lay._s, _ptr(layers.off), layers.nl, _f32(c), _f32(m),
                                _f32(v_frozen), eps, lr, p, g0, g1)


def error_norm(lay, e):
    """Per chunk, the sum of squares of the true errors e' (n_pad,) over the
    chunk's real elements, in the fixed order: (nc,) f32."""
    out = np.zeros(lay.nc, np.float32)
    lib().orc_error_norm(lay._s, _f32(e), out)
    return out


def decompress(lay, sbits, sscales, layers=None, sigma=None):
    layers = layers or Layers()
    out = np.zeros(lay.n_pad, np.float32)
    sg = None if sigma is None else _f32(sigma)
    lib().orc_decompress(lay._s, _ptr(layers.off), layers.nl, _ptr(sg),
                         np.ascontiguousarray(sbits, np.uint32), _f32(sscales), out)
    return out


def adam_update(lay, sbits, sscales, v, eps, lr, m, p):
    lib().orc_adam_update(lay._s, np.ascontiguousarray(sbits, np.uint32),
                          _f32(sscales), _f32(v), eps, lr, m, p)


def lamb_pass_a(lay, layers, sigma, sbits, sscales, v_frozen, b1, b2, m,
                v_fresh):
    R = np.zeros(layers.count(), np.float32)
    lib().orc_lamb_pass_a(lay._s, _ptr(layers.off), layers.nl, _f32(sigma),
                          np.ascontiguousarray(sbits, np.uint32), _f32(sscales),
                          _f32(v_frozen), b1, b2, m, v_fresh, R)
    return R


def lamb_ratio(R, hp, ls, frozen=False):
    """ls: dict of per-layer arrays c_avg, r_prev, c_prev, c_prev2 (updated)."""
    c = np.zeros(len(R), np.float32)
    lib().orc_lamb_ratio(len(R), _f32(R), hp["r_thr"], hp["r_min"], hp["r_max"],
                         hp["c_min"], hp["c_max"], int(frozen), ls["c_avg"],
                         ls["r_prev"], ls["c_prev"], ls["c_prev2"], c)
    return c


def lamb_pass_b(lay, layers, c, m, v_frozen, eps, lr, p):
    lib().orc_lamb_pass_b(lay._s, _ptr(layers.off), layers.nl, _f32(c), _f32(m),
                          _f32(v_frozen), eps, lr, p)


def warmup_step(lay, grads, mode, hp, m, v, p, layers=None, c_sum=None):
    """grads: list of W float32 arrays (n_pad,).  mode 0 = Adam, 1 = LAMB.
    Returns the per-layer c (LAMB) or None."""
    layers = layers or Layers()
    gs = [_f32(g) for g in grads]
    arr = (ct.c_void_p * len(gs))(*[g.ctypes.data for g in gs])
    c_out = np.zeros(layers.count(), np.float32) if mode == 1 else None
    lib().orc_warmup_step(lay._s, _ptr(layers.off), layers.nl, arr, mode,
                          hp["b1"], hp["b2"], hp["eps"], hp["lr"],
                          hp.get("c_min", 0.0), hp.get("c_max", 0.0), m, v, p,
                          _ptr(c_sum), _ptr(c_out))
    return c_out


def lamb_begin(lay, layers, m, c_sum, warmup_steps):
    L = layers.count()
    ls = {k: np.zeros(L, np.float32) for k in
          ("s", "c_avg", "r_prev", "c_prev", "c_prev2")}
    lib().orc_lamb_begin(lay._s, _ptr(layers.off), layers.nl, _f32(m),
                         _f32(c_sum), warmup_steps, ls["s"], ls["c_avg"],
                         ls["r_prev"], ls["c_prev"], ls["c_prev2"])
    return ls


def philox4x32_10(ctr, key):
    out = np.zeros(4, np.uint32)
    lib().orc_philox4x32_10(np.ascontiguousarray(ctr, np.uint32),
                            np.ascontiguousarray(key, np.uint32), out)
    return out


def uniform(seed, step, k):
    return np.float32(lib().orc_uniform(seed, step, k))


def quant_int8(g, block=256, seed=1234, step=0, deq=False, k0=0):
    """k0: index of g[0] in the whole tensor (a multiple of block)."""
    g = _f32(g)
    assert k0 % block == 0
    q = np.zeros(g.size, np.int8)
    sc = np.zeros((g.size + block - 1) // block, np.float32)
    d = np.zeros(g.size, np.float32) if deq else None
    lib().orc_quant_int8_at(g, g.size, k0, block, seed, step, q, sc, _ptr(d))
    return (q, sc, d) if deq else (q, sc)


def quant_int8_ef(g, e, seed=1234, step=0, deq=False, err2=False, k0=0):
    """INT8 (block 256) with error feedback; e is updated in place.
    Returns (q, scales[, deq][, err2])."""
    g = _f32(g)
    assert e.dtype == np.float32 and e.flags.c_contiguous and k0 % 256 == 0
    nb = (g.size + 255) // 256
    q = np.zeros(g.size, np.int8)
    sc = np.zeros(nb, np.float32)
    d = np.zeros(g.size, np.float32) if deq else None
    e2 = np.zeros(nb, np.float32) if err2 else None
    lib().orc_quant_int8_ef_at(g, e, g.size, k0, seed, step, q, sc, _ptr(d), _ptr(e2))
    out = [q, sc]
    if deq:
        out.append(d)
    if err2:
        out.append(e2)
    return tuple(out)


# ---------------------------------------------------------------------------
# Layerwise mixed bit widths: the b-bit (b = 2, 4, 8) and FP16 codecs
# ---------------------------------------------------------------------------

def qb_words(n, bits):
    """Words of packed b-bit codes for n elements (n a multiple of 256)."""
    return n * bits // 32


def qb_compress_worker(lay, bits, g, m, e, b1, w, seed, step, clip=0.0, k0=0, length=None):
    """Worker w's b-bit compression of the elements [k0, k0+length) (the
    arrays hold that range); e is updated in place.  Returns (codes u32,
    block scales f32)."""
    length = lay.n_pad - k0 if length is None else length
    assert k0 % 256 == 0 and length % 256 == 0
    assert e.dtype == np.float32 and e.flags.c_contiguous and e.size == length
    codes = np.zeros(qb_words(length, bits), np.uint32)
    sc = np.zeros(length // 256, np.float32)
    lib().orc_qb_compress_worker_at(lay._s, bits, b1, clip, w, seed, step, k0, length,
                                    _f32(g), _f32(m), e, codes, sc)
    return codes, sc


def qb_server(lay, bits, codes, bscales, e_s, seed, step, k0=0, length=None):
    """The server's b-bit average and re-compression of [k0, k0+length).
    codes: [W][words] (rows may be longer than the range: their stride is
    codes.shape[1] and they start at word k0*b/32); bscales likewise.
    e_s is updated in place.  Returns (scodes, sbscales)."""
    length = lay.n_pad - k0 if length is None else length
    assert k0 % 256 == 0 and length % 256 == 0
    assert e_s.dtype == np.float32 and e_s.flags.c_contiguous and e_s.size == length
    codes = np.ascontiguousarray(codes, np.uint32)
    bscales = _f32(bscales)
    sc = np.zeros(qb_words(length, bits), np.uint32)
    ss = np.zeros(length // 256, np.float32)
    lib().orc_qb_server_at(lay._s, bits, seed, step, k0, length, codes, codes.shape[1],
                           bscales, bscales.shape[1], e_s, sc, ss)
    return sc, ss


def qb_decode(lay, bits, codes, bscales, k0=0, length=None):
    length = lay.n_pad - k0 if length is None else length
    out = np.zeros(length, np.float32)
    lib().orc_qb_decode_at(lay._s, bits, k0, length, np.ascontiguousarray(codes, np.uint32),
                           _f32(bscales), out)
    return out


def qb_adam(lay, bits, scodes, sbscales, v, eps, lr, m, p, k0=0, length=None):
    """m, p (the range's arrays) are updated in place."""
    length = lay.n_pad - k0 if length is None else length
    lib().orc_qb_adam_at(lay._s, bits, eps, lr, k0, length,
                         np.ascontiguousarray(scodes, np.uint32), _f32(sbscales), _f32(v),
                         m, p)


def f32_to_f16(x):
    """uint16 bit patterns of IEEE binary16 (nearest, ties to even)."""
    f = lib().orc_f32_to_f16
    x = _f32(x)
    return np.array([f(float(v)) for v in x.ravel()], np.uint16).reshape(x.shape)


def f16_to_f32(h):
    f = lib().orc_f16_to_f32
    h = np.ascontiguousarray(h, np.uint16)
    return np.array([f(int(v)) for v in h.ravel()], np.float32).reshape(h.shape)


def f16_compress_worker(lay, g, m, e, b1, send, h=None, clip=0.0):
    """e is updated in place; returns h (n_pad uint16), untouched (or zeros
    if h is None) when not sending."""
    h = np.zeros(lay.n_pad, np.uint16) if h is None else h
    lib().orc_f16_compress_worker(lay._s, b1, clip, int(bool(send)), _f32(g), _f32(m), e, h)
    return h


def f16_server(lay, h, e_s):
    """h: [W][n_pad] uint16; e_s updated in place; returns hs."""
    hs = np.zeros(lay.n_pad, np.uint16)
    lib().orc_f16_server(lay._s, np.ascontiguousarray(h, np.uint16), e_s, hs)
    return hs


def f16_adam(lay, send, hs, v, eps, lr, m, p):
    lib().orc_f16_adam(lay._s, int(bool(send)), eps, lr, np.ascontiguousarray(hs, np.uint16),
                       _f32(v), m, p)


def codec_step(st, grads, hp, bits, t, seed, period=10):
    """One compressed 1-bit Adam step of a group compressed with `bits`
    (1: scaled sign, 2/4/8: block quantizer, 16: FP16 sent when t % period
    == 0), t = 1, 2, ... the compressed step.  The uniforms of the b-bit
    codec use (seed, step t)."""
    lay = st.lay
    if bits == 1:
        return compressed_step(st, grads, hp)
    clip = hp.get("clip", 0.0)
    if bits == 16:
        send = (t % period) == 0
        if not hasattr(st, "h"):
            st.h = np.zeros((lay.W, lay.n_pad), np.uint16)
            st.hs = np.zeros(lay.n_pad, np.uint16)
        for w in range(lay.W):
            f16_compress_worker(lay, grads[w], st.m, st.e[w], hp["b1"], send, st.h[w], clip)
        if send:
            st.hs = f16_server(lay, st.h, st.e_s)
        f16_adam(lay, send, st.hs, st.v, hp["eps"], hp["lr"], st.m, st.p)
        return
    codes, scs = [], []
    for w in range(lay.W):
        c, s = qb_compress_worker(lay, bits, grads[w], st.m, st.e[w], hp["b1"], w, seed, t, clip)
        codes.append(c)
        scs.append(s)
    st.codes, st.bscales = np.stack(codes), np.stack(scs)
    st.scodes, st.sbscales = qb_server(lay, bits, st.codes, st.bscales, st.e_s, seed, t)
    qb_adam(lay, bits, st.scodes, st.sbscales, st.v, hp["eps"], hp["lr"], st.m, st.p)


# ---------------------------------------------------------------------------
# Whole steps, composed from the functions above in the order of the method:
# worker compression of every worker, the server's average and
# re-compression, then the update.
# ---------------------------------------------------------------------------

class State:
    """All optimizer state of one simulated data-parallel job, on the host."""

    def __init__(self, lay, layers=None, lamb=False):
        self.lay, self.layers = lay, layers or Layers()
        z = lambda: np.zeros(lay.n_pad, np.float32)
        self.m, self.v, self.p, self.e_s = z(), z(), z(), z()
        self.e = [z() for _ in range(lay.W)]
        self.v_fresh = z() if lamb else None
        self.c_sum = np.zeros(self.layers.count(), np.float32)
        self.ls = None
        self.sbits = np.zeros(lay.words, np.uint32)
        self.sscales = np.zeros(lay.nc, np.float32)
        self.bits = np.zeros((lay.W, lay.words), np.uint32)
        self.scales = np.zeros((lay.W, lay.nc), np.float32)
        self.c = None

    def copy(self):
        import copy
        return copy.deepcopy(self)


def rho_of(ls, ratio_ef=True):
    if ls is None or not ratio_ef:
        return None
    rho = np.zeros(len(ls["c_prev"]), np.float32)
    lib().orc_lamb_rho(len(rho), _f32(ls["c_prev2"]), _f32(ls["c_prev"]), rho)
    return rho


def compressed_step(st, grads, hp, lamb=False, ratio_ef=True, frozen=False):
    """One compressed step (1-bit Adam, or 1-bit LAMB if lamb=True).
    hp["clip"] > 0 limits the workers' compensated values."""
    lay, layers = st.lay, st.layers
    sigma = st.ls["s"] if lamb else None
    rho = rho_of(st.ls, ratio_ef) if lamb else None
    for w in range(lay.W):
        b, s, _ = compress_worker(lay, grads[w], st.m, st.e[w], hp["b1"],
                                  layers, sigma, rho, hp.get("clip", 0.0))
        st.bits[w], st.scales[w] = b, s
    st.sbits, st.sscales, _ = server_reduce(lay, st.bits, st.scales, st.e_s,
                                            layers, rho)
    if not lamb:
        adam_update(lay, st.sbits, st.sscales, st.v, hp["eps"], hp["lr"], st.m,
                    st.p)
        return
    R = lamb_pass_a(lay, layers, sigma, st.sbits, st.sscales, st.v, hp["b1"],
                    hp["b2"], st.m, st.v_fresh)
    st.c = lamb_ratio(R, hp, st.ls, frozen)
    lamb_pass_b(lay, layers, st.c, st.m, st.v, hp["eps"], hp["lr"], st.p)
    st.R = R


def reset_errors(st):
    """The periodic error reset of the "1bit Adam" write-up (4.1: every 2000
    steps the compensation term is set to zero): worker and server errors."""
    for e in st.e:
        e[:] = 0
    st.e_s[:] = 0


def begin_compression(st, warmup_steps, lamb=False):
    for e in st.e:
        e[:] = 0
    st.e_s[:] = 0
    if lamb:
        st.ls = lamb_begin(st.lay, st.layers, st.m, st.c_sum, warmup_steps)
        st.v_fresh[:] = st.v
