"""bench.py's algorithmic bytes per element, checked against an explicit
list of the buffers each kernel of the step reads and writes (per real
element; G = gradient bytes, W workers, a sign word holds 32 elements).
The roofline fractions bench.py reports rest on these numbers."""
import math

import pytest

import bench

WORD = 1 / 8  # bytes of packed sign per element


def touched(W, G, lamb, sign_m):
    """Buffers per kernel: (bytes per element, times) for every read and write."""
    # sign-form m words, read per worker group (groups of 4 workers, 2 with
    # bf16 gradients; one read per tile for LAMB)
    groups = 1 if lamb else math.ceil(W / (2 if G == 2 else 4))
    compress = [(WORD, groups) if sign_m else (4, 1)]        # m
    compress += [(G, W), (4, W), (4, W), (WORD, W), (WORD, W)]  # g; e read, write; old, new word
    server = [(WORD, W), (4, 1), (4, 1), (WORD, 1), (WORD, 1)]  # worker words; e_s r/w; old, new
    if not lamb:
        update = [(WORD, 1), (4, 1), (4, 1), (4, 1)]   # sbits; v; p read, write
        if not sign_m:
            update.append((4, 1))                       # m written
    elif sign_m:
        update = [(WORD, 2), (4, 2), (4, 1)]            # A: current + previous words; v_t r/w; v_Tw
        update += [(WORD, 1), (4, 1), (4, 2)]           # B: words; v_Tw; p r/w
    else:
        update = [(WORD, 1), (4, 2), (4, 2), (4, 1)]    # A: words; m r/w; v_t r/w; v_Tw
        update += [(4, 1), (4, 1), (4, 2)]              # B: m; v_Tw; p r/w
    total = lambda xs: sum(b * k for b, k in xs)
    return {"compress": total(compress), "server": total(server), "update": total(update)}


@pytest.mark.parametrize("W,G", [(1, 4), (3, 4), (4, 2), (8, 4), (12, 2), (16, 4)])
@pytest.mark.parametrize("lamb", [False, True])
@pytest.mark.parametrize("sign_m", [False, True])
def test_bytes_per_element(W, G, lamb, sign_m):
    got = bench.bytes_per_element(W, G, lamb, sign_m)
    want = touched(W, G, lamb, sign_m)
    for k, v in want.items():
        assert got[k] == pytest.approx(v, abs=1e-12), k
    assert got["total"] == pytest.approx(sum(want.values()), abs=1e-12)


def test_headline_figures():
    """The per-element figures quoted for BERT-base (W = 8, fp32), and the
    plain count W(G + 8.25) + 28.25 (126.25 at W = 8) that leaves out the
    deferred form's re-read of the previous sign words (1/8 B per worker and
    for the server)."""
    dense = bench.bytes_per_element(8, 4, False, False)
    sign = bench.bytes_per_element(8, 4, False, True)
    assert dense["total"] == pytest.approx(127.375)
    assert dense["total"] - (8 + 1) * WORD == pytest.approx(8 * (4 + 8.25) + 28.25)
    assert sign["compress"] == pytest.approx(98.25)
    assert sign["total"] == pytest.approx(119.625)
