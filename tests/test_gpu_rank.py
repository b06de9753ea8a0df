"""The rank path (one worker and one server per process; ob_compress_worker,
ob_server_reduce_part) on one GPU: the W ranks of a job run one after
another, each with its own ctx and buffers (exchange.RankOptimizer), and
device copies stand in for the all-to-all and the all-gather -- the same
blocks exchange.py hands to the collectives.  After every compressed step
each rank's parameters, its row of words and scales, its error and its
partition of the server output equal the resident path's (all W workers in
one ctx) bit for bit, and the gathered server words and scales equal the
oracle's.  With the momentum in sign form (1-bit Adam in place, 1-bit LAMB
with the gathered output double-buffered) the ranks match the resident
path's sign form and the dense oracle all the same."""
import numpy as np
import pytest
import torch

import momentum_compression_gb300 as ob
import oracle as O
import synth
from helpers import assert_bits_equal, bf16_tensor, dev, host
from momentum_compression_gb300 import exchange as X

pytestmark = pytest.mark.gpu

f32 = np.float32
LAMB_HP = dict(b1=0.9, b2=0.999, eps=1e-6, lr=1e-3, r_thr=0.1, r_min=0.5, r_max=4.0,
               c_min=0.01, c_max=10.0)
ADAM_HP = dict(b1=0.9, b2=0.999, eps=1e-8, lr=1e-4)


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)
    from momentum_compression_gb300 import _build
    _build.build()


def _exchange(ranks, lay):
    """The all-to-all and the all-gather, by device copies."""
    wp, cpp = X.block_sizes(lay)
    W = len(ranks)
    for j, rj in enumerate(ranks):
        for w, rw in enumerate(ranks):
            rj.recv_bits[w].copy_(rw.bits_row[j * wp:(j + 1) * wp])
            rj.recv_scales[w].copy_(rw.scales_row[j * cpp:(j + 1) * cpp])


def _gather(ranks, lay):
    """The all-gather, into the buffers each rank names for this step."""
    wp, _ = X.block_sizes(lay)
    W = len(ranks)
    full_b = torch.cat([r.sbits_part for r in ranks])
    full_s = torch.cat([r.sscales_part for r in ranks])
    for r in ranks:
        sbits, sscales = r.server_targets()
        sbits[: W * wp].copy_(full_b)
        sscales.copy_(full_s)


@pytest.mark.parametrize("n,W,A,C,lamb,sign_m,dt,reset", [
    (100_003, 2, 4096, 8192, False, False, "f32", 0),
    (300_001, 4, 4096, 1 << 16, False, True, "bf16", 0),
    (50_000, 3, 128, 2048, False, True, "f32", 0),
    (70_001, 8, 128, 4096, True, False, "f32", 0),
    (40_000, 16, 128, 1024, True, False, "bf16", 0),
    (70_001, 8, 128, 4096, True, True, "f32", 0),
    (40_000, 4, 128, 1024, True, True, "bf16", 0),
    # the periodic error reset before compressed steps 3 and 5
    (100_003, 4, 128, 8192, False, True, "f32", 2),
    (70_001, 3, 128, 4096, True, True, "f32", 2),
])
def test_ranks_match_resident_path_and_oracle(n, W, A, C, lamb, sign_m, dt, reset):
    hp = LAMB_HP if lamb else ADAM_HP
    sizes = [7, 1, 4095, 4097, 33] if lamb else None
    off = None
    if lamb:
        off = [0] + list(np.cumsum(sizes))
        off.append(n)
    res = ob.OneBitOptimizer(n, W, C, A, dt, off, lamb=lamb, sign_momentum=sign_m,
                             reset_interval=reset, **hp)
    ranks = [X.RankOptimizer(n, W, r, C, A, dt, off, lamb=lamb, sign_momentum=sign_m,
                             reset_interval=reset, **hp)
             for r in range(W)]
    lay = res.layout
    wp, cpp = X.block_sizes(lay)
    P = lay["P"]
    olay = O.Layout(n, W, A, C)
    layers = O.Layers(np.array(off, np.uint64)) if lamb else None
    st = O.State(olay, layers, lamb=lamb)
    rng = np.random.default_rng(n + W)
    p0 = np.zeros(olay.n_pad, f32)
    p0[:n] = rng.standard_normal(n).astype(f32) * f32(0.02)
    st.p[:] = p0
    for o in [res] + ranks:
        o.p.copy_(torch.from_numpy(p0))

    def grads(t):
        gh, gd = [], []
        f = f32(3.0 ** -max(0, t - 2))
        for w in range(W):
            a = np.zeros(olay.n_pad, f32)
            a[:n] = rng.standard_normal(n).astype(f32) * f32(1e-3) * f
            if dt == "bf16":
                b = synth.bf16_bits(a)
                gh.append(synth.bf16_to_f32(b))
                gd.append(bf16_tensor(b))
            else:
                gh.append(a)
                gd.append(dev(a))
        return gh, gd

    warm, steps = 2, 5
    for t in range(warm):
        gh, gd = grads(t)
        res.warmup_step(gd)
        for r in ranks:
            r.warmup_step(gd)
        O.warmup_step(olay, gh, 1 if lamb else 0, hp, st.m, st.v, st.p, layers, st.c_sum)
    res.begin_compression()
    for r in ranks:
        r.begin_compression()
    O.begin_compression(st, warm, lamb=lamb)
    for t in range(warm, warm + steps):
        gh, gd = grads(t)
        res.compressed_step(gd)
        for r in ranks:
            r.begin_step()
            r.compress(gd[r.rank])
        _exchange(ranks, lay)
        for r in ranks:
            r.server()
        _gather(ranks, lay)
        for r in ranks:
            r.update()
        c = t - warm
        if reset and c and c % reset == 0:
            O.reset_errors(st)
        O.compressed_step(st, gh, hp, lamb=lamb)
        torch.cuda.synchronize()
        what = f"step {t}"
        sb = host(res.sbits)[: olay.words]
        assert_bits_equal(sb, st.sbits, f"resident server words vs oracle, {what}")
        assert_bits_equal(host(res.sscales), st.sscales, f"resident server scales vs oracle, {what}")
        for r in ranks:
            k = r.rank
            assert_bits_equal(host(r.sbits)[: olay.words], st.sbits, f"gathered words, rank {k}, {what}")
            assert_bits_equal(host(r.sscales), st.sscales, f"gathered scales, rank {k}, {what}")
            assert_bits_equal(host(r.bits_row), host(res.bits[k]), f"worker row, rank {k}, {what}")
            assert_bits_equal(host(r.scales_row), host(res.scales[k]), f"scales row, rank {k}")
            assert_bits_equal(host(r.err), host(res.err[k]), f"worker error, rank {k}, {what}")
            assert_bits_equal(host(r.err_s_part), host(res.err_s[k * P:(k + 1) * P]),
                              f"server error, partition {k}, {what}")
            assert_bits_equal(host(r.p), host(res.p), f"parameters, rank {k}, {what}")
            if lamb:
                assert_bits_equal(host(r.ls.c_t), st.c, f"c of every layer, rank {k}, {what}")
    assert_bits_equal(host(res.p)[:n], st.p[:n], "resident parameters vs oracle")
    for r in ranks:
        assert ob.ob_device_error(r.ctx) == 0
        r.close()
    res.close()


def test_server_part_rejects_unaligned_partitions():
    """P must be a multiple of 128 for the per-partition server (its word
    blocks are copied in 16-byte units); checked before any launch."""
    r = X.RankOptimizer(1064, 2, 0, 64, 32, "f32")  # P = roundup(532, 32) = 544
    assert r.layout["P"] == 544
    with pytest.raises(ob.OBError) as ei:
        r.server()
    assert ei.value.status == ob.OB_ERR_UNSUPPORTED
    assert "multiple of 128" in ob.ob_last_error(r.ctx)
    r.close()
