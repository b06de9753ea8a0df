"""One compressed step of the oracle over a whole fused buffer, run as
independent chunk ranges on a thread pool.

The oracle's compressed step is chunk-local: every output element depends
only on the inputs of its own chunk, except 1-bit LAMB's per-layer maximum
ratio R_l, a maximum over the layer.  So the step is split into one range
of chunks per partition (the W partitions' boundaries fall on multiples of
32 elements when the alignment does), each stage's ranges run in parallel
threads (the oracle's C calls release the GIL), the ranges' R are merged by
maximum, and the per-layer ratio update runs once.  The result is the
oracle's whole-buffer step bit for bit (tests/test_oracle_ranges.py checks
that); it only takes a fraction of the time on whole-model sizes.
"""
import numpy as np

import oracle as O


def partition_ranges(lay):
    """[(g0, g1)] chunk ranges, one per partition."""
    return [(j * lay.cpp, (j + 1) * lay.cpp) for j in range(lay.W)]


def compressed_step(st, grads, hp, pool, lamb=False, ratio_ef=True, frozen=False):
    """O.compressed_step(st, grads, hp, lamb, ratio_ef, frozen), with the
    same calls in the same order, each split over the partitions' chunk
    ranges and run on `pool` (a concurrent.futures executor)."""
    lay, layers = st.lay, st.layers
    rngs = partition_ranges(lay)
    sigma = st.ls["s"] if lamb else None
    rho = O.rho_of(st.ls, ratio_ef) if lamb else None
    st.bits = np.zeros((lay.W, lay.words), np.uint32)
    st.scales = np.zeros((lay.W, lay.nc), np.float32)
    jobs = [pool.submit(O.compress_worker_range, lay, g0, g1, grads[w], st.m, st.e[w],
                        st.bits[w], st.scales[w], hp["b1"], layers, sigma, rho,
                        hp.get("clip", 0.0))
            for w in range(lay.W) for g0, g1 in rngs]
    for j in jobs:
        j.result()
    st.sbits = np.zeros(lay.words, np.uint32)
    st.sscales = np.zeros(lay.nc, np.float32)
    jobs = [pool.submit(O.server_reduce_range, lay, g0, g1, st.bits, st.scales, st.e_s,
                        st.sbits, st.sscales, layers, rho) for g0, g1 in rngs]
    for j in jobs:
        j.result()
    if not lamb:
        O.adam_update(lay, st.sbits, st.sscales, st.v, hp["eps"], hp["lr"], st.m, st.p)
        return
    jobs = [pool.submit(O.lamb_pass_a_range, lay, g0, g1, layers, sigma, st.sbits, st.sscales,
                        st.v, hp["b1"], hp["b2"], st.m, st.v_fresh) for g0, g1 in rngs]
    R = np.zeros(layers.count(), np.float32)
    for j in jobs:
        R = np.maximum(R, j.result())
    st.c = O.lamb_ratio(R, hp, st.ls, frozen)
    jobs = [pool.submit(O.lamb_pass_b_range, lay, g0, g1, layers, st.c, st.m, st.v, hp["eps"],
                        hp["lr"], st.p) for g0, g1 in rngs]
    for j in jobs:
        j.result()
    st.R = R
