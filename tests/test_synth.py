"""The synthetic workloads: parameter counts of the model lists (the
published sizes of these architectures) and the grouping by bit width for
layerwise mixed widths.  CPU only."""
import numpy as np

import synth


def test_model_sizes():
    for fn, count, total in [(synth.bert_base_tensors, 199, 109_482_240),
                             (synth.bert_large_tensors, 302, 336_226_108),
                             (synth.gpt_1p3b_tensors, 292, 1_315_723_264)]:
        t = fn()
        assert len(t) == count and sum(s for _, s, _ in t) == total


def test_resnet50_size():
    """torchvision's ResNet-50: 161 parameter tensors, 25,557,032 values, of
    which 53 convolutions and 53 batch norms."""
    p = synth.resnet50_params()
    assert len(p) == 161 and sum(x[1] for x in p) == 25_557_032
    assert sum(x[3] == "conv" for x in p) == 53
    assert sum(x[3] == "norm" for x in p) == 106
    assert sum(x[1] for x in p if x[3] == "norm") == 2 * 26_560


def test_mixed_groups_partition_the_model_in_order():
    p = synth.resnet50_params()
    groups = synth.mixed_groups()
    assert [b for b, _ in groups] == [1, 2, 16]
    names = []
    for bits, wl in groups:
        assert all(synth.LAYERWISE_BITS[q[3]] == bits
                   for q in p if q[0] in {t[0] for t in wl.tensors})
        assert wl.n == sum(s for _, s, _ in wl.tensors) and wl.seed_tag == bits
        order = [q[0] for q in p if synth.LAYERWISE_BITS[q[3]] == bits]
        assert [t[0] for t in wl.tensors] == order
        names += order
    assert sorted(names) == sorted(q[0] for q in p)
    assert sum(wl.n for _, wl in groups) == 25_557_032


def test_groups_draw_from_separate_streams():
    (_, a), (_, b) = synth.mixed_groups()[:2]
    ga = synth.grad_slice(a, 0, 0, 0, 4096) / synth._std_per_element(a, 0, 4096)
    gb = synth.grad_slice(b, 0, 0, 0, 4096) / synth._std_per_element(b, 0, 4096)
    assert not np.allclose(ga, gb)
    c = synth.workload("flat", n=4096, W=1, chunk=4096)
    gc = synth.grad_slice(c, 0, 0, 0, 4096) / np.float32(1e-3)
    assert not np.allclose(ga, gc)
