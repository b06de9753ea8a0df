"""The oracle's chunk-range functions against its whole-buffer functions.

Every whole-buffer 1-bit function of the oracle is its range function over
all chunks; these tests check the other direction: splitting the chunks
into ranges (at the partitions, and at arbitrary chunk boundaries), run
one after the other or in concurrent threads, gives the whole-buffer
results bit for bit -- sign words, scales, errors, momentum, fresh
variance, LAMB's R and c, and parameters.  That is what lets the
full-size parity tests run the oracle on a whole model in parallel
(tests/oracle_parallel.py).  CPU only.
"""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

import oracle as O
import oracle_parallel as OP

f32 = np.float32

HP = dict(b1=0.9, b2=0.999, eps=1e-6, lr=1e-3, r_thr=0.1, r_min=0.5, r_max=4.0, c_min=0.01,
          c_max=10.0)


def _state(n, W, A, C, sizes, lamb, seed):
    rng = np.random.default_rng(seed)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.uint64) if sizes else None
    lay = O.Layout(n, W, A, C)
    layers = O.Layers(off)
    st = O.State(lay, layers, lamb=lamb)
    st.m[:n] = rng.standard_normal(n).astype(f32) * f32(1e-3)
    st.v[:n] = np.abs(rng.standard_normal(n)).astype(f32) * f32(1e-6) + f32(1e-12)
    st.p[:n] = rng.standard_normal(n).astype(f32) * f32(0.02)
    st.e_s[:n] = rng.standard_normal(n).astype(f32) * f32(1e-4)
    for e in st.e:
        e[:n] = rng.standard_normal(n).astype(f32) * f32(1e-4)
    if lamb:
        st.v_fresh[:] = st.v
        L = layers.count()
        st.ls = {"s": (10.0 ** rng.uniform(-1, 1, L)).astype(f32),
                 "c_avg": (10.0 ** rng.uniform(-0.5, 0.5, L)).astype(f32),
                 "r_prev": np.ones(L, f32)}
        st.ls["c_prev"] = (st.ls["c_avg"] * f32(1.05)).astype(f32)
        st.ls["c_prev2"] = st.ls["c_avg"].copy()
    grads = []
    for t in range(4):
        gs = []
        for w in range(W):
            a = np.zeros(lay.n_pad, f32)
            a[:n] = rng.standard_normal(n).astype(f32) * f32(1e-3 * 3.0 ** -t)
            gs.append(a)
        grads.append(gs)
    return st, grads


def _same(a, b, what):
    a, b = np.ascontiguousarray(a), np.ascontiguousarray(b)
    assert a.shape == b.shape, what
    assert np.array_equal(a.view(np.uint32) if a.dtype == f32 else a,
                          b.view(np.uint32) if b.dtype == f32 else b), what


def _compare(st_a, st_b, lamb):
    _same(st_a.bits, st_b.bits, "worker sign words")
    _same(st_a.scales, st_b.scales, "worker scales")
    _same(st_a.sbits, st_b.sbits, "server sign words")
    _same(st_a.sscales, st_b.sscales, "server scales")
    for w, (x, y) in enumerate(zip(st_a.e, st_b.e)):
        _same(x, y, f"error of worker {w}")
    for k in ("e_s", "m", "p"):
        _same(getattr(st_a, k), getattr(st_b, k), k)
    if lamb:
        _same(st_a.v_fresh, st_b.v_fresh, "v_fresh")
        _same(st_a.R, st_b.R, "R")
        _same(st_a.c, st_b.c, "c")
        for k in ("r_prev", "c_prev", "c_prev2"):
            _same(st_a.ls[k], st_b.ls[k], k)


@pytest.mark.parametrize("n,W,A,C,sizes", [
    (100_003, 4, 4096, 8192, [7, 1, 2, 4095, 4097, 33, 1000, 20000, 3, 70765]),
    (50_001, 3, 32, 2048, [50_001]),
    (3 * 4096 + 5, 8, 32, 96, [5, 4096, 2, 4096, 4092, 2]),
    (1, 1, 32, 32, [1]),
])
@pytest.mark.parametrize("lamb", [False, True])
def test_threaded_partition_step_equals_whole_step(n, W, A, C, sizes, lamb):
    """Four compressed steps of the oracle, whole-buffer and split into one
    range per partition on 8 threads: identical state after every step."""
    st_a, grads = _state(n, W, A, C, sizes, lamb, seed=n + W)
    st_b, _ = _state(n, W, A, C, sizes, lamb, seed=n + W)
    with ThreadPoolExecutor(8) as pool:
        for t in range(4):
            O.compressed_step(st_a, grads[t], HP, lamb=lamb)
            OP.compressed_step(st_b, grads[t], HP, pool, lamb=lamb)
            _compare(st_a, st_b, lamb)


def test_arbitrary_chunk_ranges_equal_whole():
    """Ranges cut at arbitrary chunk boundaries (not only at partitions),
    run one after the other, for each range function."""
    n, W, A, C = 70_001, 3, 4096, 2048
    sizes = [3, 4097, 30_000, 5, 35_896]
    st, grads = _state(n, W, A, C, sizes, True, seed=5)
    lay, layers = st.lay, st.layers
    rho = O.rho_of(st.ls)
    cuts = [0, 1, 4, 5, 11, lay.nc]
    for w in range(W):
        e_a, e_b = st.e[w].copy(), st.e[w].copy()
        bits_a, sc_a, _ = O.compress_worker(lay, grads[0][w], st.m, e_a, HP["b1"], layers,
                                            st.ls["s"], rho)
        bits_b = np.zeros(lay.words, np.uint32)
        sc_b = np.zeros(lay.nc, f32)
        for g0, g1 in zip(cuts[:-1], cuts[1:]):
            O.compress_worker_range(lay, g0, g1, grads[0][w], st.m, e_b, bits_b, sc_b, HP["b1"],
                                    layers, st.ls["s"], rho)
        _same(bits_b, bits_a, "bits")
        _same(sc_b, sc_a, "scales")
        _same(e_b, e_a, "errors")
        st.bits[w], st.scales[w] = bits_a, sc_a
    es_a, es_b = st.e_s.copy(), st.e_s.copy()
    sb_a, ss_a, _ = O.server_reduce(lay, st.bits, st.scales, es_a, layers, rho)
    sb_b = np.zeros(lay.words, np.uint32)
    ss_b = np.zeros(lay.nc, f32)
    for g0, g1 in zip(cuts[:-1], cuts[1:]):
        O.server_reduce_range(lay, g0, g1, st.bits, st.scales, es_b, sb_b, ss_b, layers, rho)
    _same(sb_b, sb_a, "sbits")
    _same(ss_b, ss_a, "sscales")
    _same(es_b, es_a, "e_s")
    m_a, m_b = st.m.copy(), st.m.copy()
    vf_a, vf_b = st.v_fresh.copy(), st.v_fresh.copy()
    R_a = O.lamb_pass_a(lay, layers, st.ls["s"], sb_a, ss_a, st.v, HP["b1"], HP["b2"], m_a, vf_a)
    R_b = np.zeros_like(R_a)
    for g0, g1 in zip(cuts[:-1], cuts[1:]):
        R_b = np.maximum(R_b, O.lamb_pass_a_range(lay, g0, g1, layers, st.ls["s"], sb_b, ss_b,
                                                  st.v, HP["b1"], HP["b2"], m_b, vf_b))
    _same(R_b, R_a, "R")
    _same(m_b, m_a, "m")
    _same(vf_b, vf_a, "v_fresh")
    c = (10.0 ** np.linspace(-1, 1, layers.count())).astype(f32)
    p_a, p_b = st.p.copy(), st.p.copy()
    O.lamb_pass_b(lay, layers, c, m_a, st.v, HP["eps"], HP["lr"], p_a)
    for g0, g1 in zip(cuts[:-1], cuts[1:]):
        O.lamb_pass_b_range(lay, g0, g1, layers, c, m_b, st.v, HP["eps"], HP["lr"], p_b)
    _same(p_b, p_a, "p")
