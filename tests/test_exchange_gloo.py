"""The rank path's two collectives (momentum_compression_gb300/exchange.py)
on the CPU with gloo, world size 2: the all-to-all of the compressed
blocks and the all-gather of the servers' outputs, with words and scales
made by the oracle (no GPU).

Each rank runs the oracle's compression for every worker from the same
seeded gradients, sends its own row, and checks that it received exactly
partition `rank` of every worker's row, in rank order; that the oracle's
server run on those received blocks alone (chunk range of its partition)
gives the whole-buffer server's output for that partition; and that the
all-gather of the partitions' outputs is the whole server output.  Two
steps, so the errors carried between them are not zero."""
import os
import socket
import sys

import numpy as np
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

N, WORLD, A, C = 20_001, 2, 128, 1024


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch
    import torch.distributed as dist

    import momentum_compression_gb300 as ob
    import oracle as O
    from momentum_compression_gb300 import exchange as X
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        ctx = ob.ob_init(N, WORLD, C, A)  # host only: the layout the ranks share
        lay = ob.ob_get_layout(ctx)
        ob.ob_destroy(ctx)
        olay = O.Layout(N, WORLD, A, C)
        assert (lay["n_pad"], lay["P"], lay["n_chunks"]) == (olay.n_pad, olay.P, olay.nc)
        wp, cpp = X.block_sizes(lay)
        rng = np.random.default_rng(77)
        st = O.State(olay)
        st.m[:N] = rng.standard_normal(N).astype(np.float32) * np.float32(1e-3)
        for step in range(2):
            grads = []
            for w in range(WORLD):
                a = np.zeros(olay.n_pad, np.float32)
                a[:N] = rng.standard_normal(N).astype(np.float32) * np.float32(1e-3)
                grads.append(a)
            bits = np.zeros((WORLD, olay.words), np.uint32)
            scales = np.zeros((WORLD, olay.nc), np.float32)
            for w in range(WORLD):
                bits[w], scales[w], _ = O.compress_worker(olay, grads[w], st.m, st.e[w], 0.9)
            # this rank's row, in the device row layout (words rounded up to 4)
            row = torch.zeros(lay["words_per_worker"], dtype=torch.int32)
            row[: olay.words] = torch.from_numpy(bits[rank].view(np.int32))
            srow = torch.from_numpy(scales[rank].copy())
            recv_bits = torch.zeros((WORLD, wp), dtype=torch.int32)
            recv_scales = torch.zeros((WORLD, cpp), dtype=torch.float32)
            X.exchange_worker_blocks(row, srow, lay, recv_bits, recv_scales)
            rb = recv_bits.numpy().view(np.uint32)
            for w in range(WORLD):
                assert np.array_equal(rb[w], bits[w][rank * wp:(rank + 1) * wp]), (step, w)
                assert np.array_equal(recv_scales[w].numpy(),
                                      scales[w][rank * cpp:(rank + 1) * cpp]), (step, w)
            # the whole-buffer server, and this rank's partition from the
            # received blocks alone
            es_part = st.e_s[rank * olay.P:(rank + 1) * olay.P].copy()
            sbits, sscales, _ = O.server_reduce(olay, bits, scales, st.e_s)
            only = np.zeros_like(bits)
            only_sc = np.zeros_like(scales)
            for w in range(WORLD):
                only[w][rank * wp:(rank + 1) * wp] = rb[w]
                only_sc[w][rank * cpp:(rank + 1) * cpp] = recv_scales[w].numpy()
            es_full = np.zeros(olay.n_pad, np.float32)
            es_full[rank * olay.P:(rank + 1) * olay.P] = es_part
            sb_p = np.zeros(olay.words, np.uint32)
            ss_p = np.zeros(olay.nc, np.float32)
            O.server_reduce_range(olay, rank * cpp, (rank + 1) * cpp, only, only_sc, es_full,
                                  sb_p, ss_p)
            assert np.array_equal(sb_p[rank * wp:(rank + 1) * wp],
                                  sbits[rank * wp:(rank + 1) * wp]), step
            assert np.array_equal(ss_p[rank * cpp:(rank + 1) * cpp],
                                  sscales[rank * cpp:(rank + 1) * cpp]), step
            assert np.array_equal(es_full[rank * olay.P:(rank + 1) * olay.P],
                                  st.e_s[rank * olay.P:(rank + 1) * olay.P]), step
            # the all-gather of the partitions' outputs
            part_b = torch.from_numpy(sb_p[rank * wp:(rank + 1) * wp].view(np.int32).copy())
            part_s = torch.from_numpy(ss_p[rank * cpp:(rank + 1) * cpp].copy())
            all_b = torch.zeros(lay["words_per_worker"], dtype=torch.int32)
            all_s = torch.zeros(lay["n_chunks"], dtype=torch.float32)
            X.gather_server(part_b, part_s, lay, all_b, all_s)
            assert np.array_equal(all_b.numpy().view(np.uint32)[: olay.words], sbits), step
            assert np.array_equal(all_s.numpy(), sscales), step
            O.adam_update(olay, sbits, sscales, np.ones(olay.n_pad, np.float32), 1e-8, 1e-4,
                          st.m, st.p)
        out.put((rank, "ok"))
    except Exception as e:  # reported to the test process
        out.put((rank, repr(e)))
        raise
    finally:
        dist.destroy_process_group()


def test_exchange_layout_world_size_2_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, port, q)) for r in range(WORLD)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
    assert res == [(0, "ok"), (1, "ok")], res
    assert all(p.exitcode == 0 for p in procs)
