"""Seeded synthetic workloads for the 1-bit compressed optimizer step.

The pages measure on BERT-base / BERT-large pre-training, GPT-style models,
ResNet-50 and ImageNet; none of that data or those weights are available,
so these generators stand in for them: parameter lists with the models'
exact tensor shapes fused into one 1-D buffer, Gaussian gradients whose
standard deviation varies per tensor, and initial parameters drawn the way
such models are initialised.

This module is shared by the tests (for both the CUDA path and the oracle)
and by bench.py.  It holds none of the method's arithmetic: it only draws
numbers.  Gradient values for any slice of the fused buffer can be drawn
independently, because each block of BLOCK elements has its own seed.
"""
from dataclasses import dataclass, field
from typing import List, Optional, Tuple

import numpy as np

SEED_BASE = 1234
BLOCK = 1 << 20


# ---------------------------------------------------------------------------
# Parameter lists (name, numel, kind); kind decides the initial value:
# "w" ~ N(0, 0.02), "ln_w" = 1, "b" = 0.
# ---------------------------------------------------------------------------

def bert_base_tensors() -> List[Tuple[str, int, str]]:
    """BERT-base (hidden 768, FFN 3072, 12 layers, vocab 30522, 512
    positions, 2 token types, pooler): 199 tensors, 109,482,240 values."""
    h, f, L = 768, 3072, 12
    t = [("emb.word", 30522 * h, "w"), ("emb.pos", 512 * h, "w"),
         ("emb.type", 2 * h, "w"), ("emb.ln.w", h, "ln_w"), ("emb.ln.b", h, "b")]
    for i in range(L):
        p = f"l{i}."
        for q in ("q", "k", "v"):
            t += [(p + q + ".w", h * h, "w"), (p + q + ".b", h, "b")]
        t += [(p + "o.w", h * h, "w"), (p + "o.b", h, "b"),
              (p + "ln1.w", h, "ln_w"), (p + "ln1.b", h, "b"),
              (p + "fc1.w", h * f, "w"), (p + "fc1.b", f, "b"),
              (p + "fc2.w", f * h, "w"), (p + "fc2.b", h, "b"),
              (p + "ln2.w", h, "ln_w"), (p + "ln2.b", h, "b")]
    t += [("pool.w", h * h, "w"), ("pool.b", h, "b")]
    return t


def bert_large_tensors() -> List[Tuple[str, int, str]]:
    """BERT-large with fused QKV (hidden 1024, FFN 4096, 24 layers), MLM
    head (dense, LayerNorm, decoder bias; decoder weight tied) and NSP head:
    302 tensors, 336,226,108 values (the 302 matches the per-layer
    collective count the 1-bit LAMB summary gives for BERT-Large)."""
    h, f, L, V = 1024, 4096, 24, 30522
    t = [("emb.word", V * h, "w"), ("emb.pos", 512 * h, "w"),
         ("emb.type", 2 * h, "w"), ("emb.ln.w", h, "ln_w"), ("emb.ln.b", h, "b")]
    for i in range(L):
        p = f"l{i}."
        t += [(p + "qkv.w", h * 3 * h, "w"), (p + "qkv.b", 3 * h, "b"),
              (p + "o.w", h * h, "w"), (p + "o.b", h, "b"),
              (p + "ln1.w", h, "ln_w"), (p + "ln1.b", h, "b"),
              (p + "fc1.w", h * f, "w"), (p + "fc1.b", f, "b"),
              (p + "fc2.w", f * h, "w"), (p + "fc2.b", h, "b"),
              (p + "ln2.w", h, "ln_w"), (p + "ln2.b", h, "b")]
    t += [("pool.w", h * h, "w"), ("pool.b", h, "b"),
          ("mlm.dense.w", h * h, "w"), ("mlm.dense.b", h, "b"),
          ("mlm.ln.w", h, "ln_w"), ("mlm.ln.b", h, "b"), ("mlm.dec.b", V, "b"),
          ("nsp.w", h * 2, "w"), ("nsp.b", 2, "b")]
    return t


def gpt_1p3b_tensors() -> List[Tuple[str, int, str]]:
    """GPT with 24 layers, hidden 2048, FFN 8192, vocab 50257, context 2048:
    292 tensors, 1,315,723,264 values."""
    h, f, L, V, T = 2048, 8192, 24, 50257, 2048
    t = [("wte", V * h, "w"), ("wpe", T * h, "w")]
    for i in range(L):
        p = f"l{i}."
        t += [(p + "ln1.w", h, "ln_w"), (p + "ln1.b", h, "b"),
              (p + "qkv.w", h * 3 * h, "w"), (p + "qkv.b", 3 * h, "b"),
              (p + "proj.w", h * h, "w"), (p + "proj.b", h, "b"),
              (p + "ln2.w", h, "ln_w"), (p + "ln2.b", h, "b"),
              (p + "fc.w", h * f, "w"), (p + "fc.b", f, "b"),
              (p + "proj2.w", f * h, "w"), (p + "proj2.b", h, "b")]
    t += [("lnf.w", h, "ln_w"), ("lnf.b", h, "b")]
    return t


def resnet50_params() -> List[Tuple[str, int, str, str]]:
    """ResNet-50 (bottleneck blocks 3-4-6-3, widths 64-128-256-512, expansion
    4, 1000 classes) as (name, numel, init kind, parameter type): 53
    convolutions, 53 batch norms (weight and bias), the fc layer: 161
    tensors, 25,557,032 values.  Types: "conv", "norm", "dense"."""
    t = []

    def conv(name, cin, cout, k):
        t.append((name + ".weight", cin * cout * k * k, "w", "conv"))

    def bn(name, c):
        t.extend([(name + ".weight", c, "ln_w", "norm"), (name + ".bias", c, "b", "norm")])

    conv("conv1", 3, 64, 7)
    bn("bn1", 64)
    cin = 64
    for li, (mid, blocks) in enumerate([(64, 3), (128, 4), (256, 6), (512, 3)], 1):
        out = 4 * mid
        for b in range(blocks):
            pre = f"layer{li}.{b}"
            conv(pre + ".conv1", cin, mid, 1)
            bn(pre + ".bn1", mid)
            conv(pre + ".conv2", mid, mid, 3)
            bn(pre + ".bn2", mid)
            conv(pre + ".conv3", mid, out, 1)
            bn(pre + ".bn3", out)
            if b == 0:
                conv(pre + ".downsample.0", cin, out, 1)
                bn(pre + ".downsample.1", out)
            cin = out
    t.extend([("fc.weight", 2048 * 1000, "w", "dense"), ("fc.bias", 1000, "b", "dense")])
    return t


# Bit width per parameter type for layerwise mixed widths: embeddings and
# dense (transformer FFN) layers 1 bit, convolution weights 2 bits,
# normalisation parameters FP16 sent every NORM_PERIOD-th step (the "1bit
# Adam" write-up, §3.2 table and §6 layerwise_bits [1, 2, 1, 16]).
LAYERWISE_BITS = {"embedding": 1, "conv": 2, "dense": 1, "norm": 16}
NORM_PERIOD = 10


# ---------------------------------------------------------------------------
# Workloads
# ---------------------------------------------------------------------------

@dataclass
class Workload:
    name: str
    n: int
    W: int
    chunk: int
    align: int = 4096
    grad_dtype: str = "f32"          # "f32" or "bf16"
    mode: str = "adam"               # "adam" or "lamb"
    tensors: Optional[List[Tuple[str, int, str]]] = None
    layer_std: Optional[np.ndarray] = None   # per tensor, float64
    flat_std: float = 1e-3
    std_decay: float = 1.0           # std factor reached at the last compressed step
    warmup_steps: int = 5
    compressed_steps: int = 10
    hp: dict = field(default_factory=dict)
    seed_tag: int = 0                # != 0: a separate family of random streams

    @property
    def layer_offsets(self) -> Optional[np.ndarray]:
        if self.tensors is None:
            return None
        sizes = np.array([s for _, s, _ in self.tensors], dtype=np.uint64)
        return np.concatenate([[0], np.cumsum(sizes)]).astype(np.uint64)

    @property
    def n_layers(self) -> int:
        return 0 if self.tensors is None else len(self.tensors)

    def std_factor(self, step: int) -> float:
        """Gradient std factor at `step` (warmup steps are numbered
        0..warmup-1, compressed steps follow).  For the LAMB workload the std
        decays geometrically by `std_decay` over the compressed steps, so the
        fresh variance falls by its square (the 1-bit LAMB summary: per-layer
        variance norms keep falling by up to two orders of magnitude)."""
        t = step - self.warmup_steps
        if t <= 0 or self.std_decay == 1.0 or self.compressed_steps <= 1:
            return 1.0
        t = min(t, self.compressed_steps - 1)
        return float(self.std_decay ** (t / (self.compressed_steps - 1)))


ADAM_HP = dict(b1=0.9, b2=0.999, eps=1e-8, lr=1e-4)


def _tensor_std(tensors, seed=SEED_BASE):
    rng = np.random.default_rng(np.random.SeedSequence([seed, 7]))
    return 1e-3 * 10.0 ** rng.uniform(-1.0, 1.0, size=len(tensors))


def workload(name: str, **over) -> Workload:
    """Named workloads:
    flat-1m    : n = 2^20, W = 4, chunk 2^18, 1-bit Adam, 5 + 10 steps
    bert-base  : BERT-base list, W = 8, chunk 2^20, 1-bit Adam, 100 + 50 steps
    bert-large : BERT-large list, W = 8, chunk 2^20, 1-bit LAMB, 100 + 50
                 steps, gradient std decaying 10x over the compressed steps
    gpt-1.3b   : GPT-1.3B list, W = 4, bf16 gradients, chunk 2^20, 1-bit Adam,
                 5 + 10 steps
    flat       : the bandwidth sweep point; pass n, W, chunk
    """
    if name == "flat-1m":
        wl = Workload(name, n=1 << 20, W=4, chunk=1 << 18, hp=dict(ADAM_HP))
    elif name == "bert-base":
        t = bert_base_tensors()
        wl = Workload(name, n=sum(s for _, s, _ in t), W=8, chunk=1 << 20,
                      tensors=t, layer_std=_tensor_std(t), warmup_steps=100,
                      compressed_steps=50, hp=dict(ADAM_HP))
    elif name == "bert-large":
        t = bert_large_tensors()
        hp = dict(b1=0.9, b2=0.999, eps=1e-6, lr=1e-3, r_thr=0.1, r_min=0.5,
                  r_max=4.0, c_min=0.01, c_max=10.0)
        wl = Workload(name, n=sum(s for _, s, _ in t), W=8, chunk=1 << 20,
                      mode="lamb", tensors=t, layer_std=_tensor_std(t),
                      std_decay=0.1, warmup_steps=100, compressed_steps=50, hp=hp)
    elif name == "gpt-1.3b":
        t = gpt_1p3b_tensors()
        wl = Workload(name, n=sum(s for _, s, _ in t), W=4, chunk=1 << 20,
                      grad_dtype="bf16", tensors=t, layer_std=_tensor_std(t),
                      warmup_steps=5, compressed_steps=10, hp=dict(ADAM_HP))
    elif name == "flat":
        wl = Workload(name, n=over.pop("n"), W=over.pop("W"),
                      chunk=over.pop("chunk"), hp=dict(ADAM_HP))
    else:
        raise KeyError(name)
    for k, v in over.items():
        if k in ("hp",):
            wl.hp.update(v)
        else:
            setattr(wl, k, v)
    return wl


def mixed_groups(name: str = "resnet50-mixed", W: int = 8, warmup_steps: int = 5,
                 compressed_steps: int = 20) -> List[Tuple[int, Workload]]:
    """Layerwise mixed widths: the model's tensors grouped by the bit width
    of their type (LAYERWISE_BITS), each group a fused buffer of its own
    (tensors in model order), as [(bits, Workload)] in increasing width.
    Per-tensor gradient std 1e-3*10^U(-1,1) drawn over the whole model;
    each group draws from its own random streams (seed_tag = bits)."""
    if name != "resnet50-mixed":
        raise KeyError(name)
    params = resnet50_params()
    std = _tensor_std(params)
    groups = []
    for bits in sorted(set(LAYERWISE_BITS[p[3]] for p in params)):
        idx = [i for i, p in enumerate(params) if LAYERWISE_BITS[p[3]] == bits]
        t = [params[i][:3] for i in idx]
        wl = Workload(f"{name}/{bits}", n=sum(s for _, s, _ in t), W=W, chunk=1 << 20,
                      tensors=t, layer_std=std[idx], warmup_steps=warmup_steps,
                      compressed_steps=compressed_steps, hp=dict(ADAM_HP), seed_tag=bits)
        groups.append((bits, wl))
    return groups


# ---------------------------------------------------------------------------
# Drawing numbers
# ---------------------------------------------------------------------------

def _tag(wl: Workload) -> list:
    return [wl.seed_tag] if wl.seed_tag else []


def _std_per_element(wl: Workload, start: int, stop: int) -> np.ndarray:
    """float32 std for elements [start, stop) (0 beyond n)."""
    out = np.zeros(stop - start, np.float32)
    hi = min(stop, wl.n)
    if hi <= start:
        return out
    if wl.tensors is None:
        out[: hi - start] = wl.flat_std
        return out
    off = wl.layer_offsets.astype(np.int64)
    l0 = int(np.searchsorted(off, start, side="right") - 1)
    l1 = int(np.searchsorted(off, hi - 1, side="right") - 1)
    for l in range(l0, l1 + 1):
        a, b = max(int(off[l]), start), min(int(off[l + 1]), hi)
        out[a - start: b - start] = wl.layer_std[l]
    return out


def grad_slice(wl: Workload, step: int, worker: int, start: int,
               stop: int) -> np.ndarray:
    """float32 gradient values of `worker` at `step` for elements
    [start, stop); elements >= n are 0.  Gradient seed = SEED_BASE +
    1000*step + worker, one independent stream per block of BLOCK elements."""
    out = np.empty(stop - start, np.float32)
    b0, b1 = start // BLOCK, (stop - 1) // BLOCK if stop > start else -1
    for b in range(b0, b1 + 1):
        ss = np.random.SeedSequence([SEED_BASE + 1000 * step + worker, b] + _tag(wl))
        z = np.random.default_rng(ss).standard_normal(BLOCK, dtype=np.float32)
        a, c = max(b * BLOCK, start), min((b + 1) * BLOCK, stop)
        out[a - start: c - start] = z[a - b * BLOCK: c - b * BLOCK]
    std = _std_per_element(wl, start, stop) * np.float32(wl.std_factor(step))
    out *= std
    return out


def params0_slice(wl: Workload, start: int, stop: int) -> np.ndarray:
    """Initial parameters: weights N(0, 0.02), LayerNorm weights 1, biases
    0 (flat workloads: all N(0, 0.02)); 0 beyond n."""
    out = np.empty(stop - start, np.float32)
    b0, b1 = start // BLOCK, (stop - 1) // BLOCK if stop > start else -1
    for b in range(b0, b1 + 1):
        ss = np.random.SeedSequence([SEED_BASE, 999_999, b] + _tag(wl))
        z = np.random.default_rng(ss).standard_normal(BLOCK, dtype=np.float32)
        a, c = max(b * BLOCK, start), min((b + 1) * BLOCK, stop)
        out[a - start: c - start] = z[a - b * BLOCK: c - b * BLOCK]
    out *= np.float32(0.02)
    hi = min(stop, wl.n)
    out[max(hi - start, 0):] = 0.0
    if wl.tensors is not None and hi > start:
        off = wl.layer_offsets.astype(np.int64)
        l0 = int(np.searchsorted(off, start, side="right") - 1)
        l1 = int(np.searchsorted(off, hi - 1, side="right") - 1)
        for l in range(l0, l1 + 1):
            kind = wl.tensors[l][2]
            if kind == "w":
                continue
            a, b = max(int(off[l]), start), min(int(off[l + 1]), hi)
            out[a - start: b - start] = 1.0 if kind == "ln_w" else 0.0
    return out


def state_slice(wl: Workload, what: str, start: int, stop: int,
                worker: int = 0) -> np.ndarray:
    """Directly initialised compressed-phase state for sweep points (no
    warmup): m and e ~ N(0, 1e-3), v ~ |N(0, 1e-6)| + 1e-12; 0 beyond n."""
    tag = {"m": 1, "e": 2, "v": 3, "e_s": 4}[what]
    out = np.empty(stop - start, np.float32)
    b0, b1 = start // BLOCK, (stop - 1) // BLOCK if stop > start else -1
    for b in range(b0, b1 + 1):
        ss = np.random.SeedSequence([SEED_BASE, 500_000 + tag, worker, b] + _tag(wl))
        z = np.random.default_rng(ss).standard_normal(BLOCK, dtype=np.float32)
        a, c = max(b * BLOCK, start), min((b + 1) * BLOCK, stop)
        out[a - start: c - start] = z[a - b * BLOCK: c - b * BLOCK]
    if what == "v":
        out = np.abs(out) * np.float32(1e-6) + np.float32(1e-12)
    else:
        out *= np.float32(1e-3)
    hi = min(stop, wl.n)
    out[max(hi - start, 0):] = 0.0
    return out


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns the uint16
    bit patterns.  NaN is kept as a quiet NaN."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    r = ((u >> 16) & 1) + 0x7FFF
    out = ((u + r) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)
