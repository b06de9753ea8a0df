"""Throughput of the fused 1-bit compressed optimizer step on GB300.

One step = worker compression of all W workers (ob_compress), the server
average and re-compression (ob_server_reduce) and the unpack + frozen
variance update (ob_adam_step, or ob_lamb_step for 1-bit LAMB).  The
headline workload is the largest single-GPU one: the GPT-1.3B-shaped list
(1,315,723,264 parameters in 292 tensors fused into one buffer), bf16
gradients, fp32 state, W = 4 simulated data-parallel workers, chunk 2^20.
Inputs are resident in HBM (about 92 GB touched per step, far above the
129 MB L2, so no flush is needed).

Prints ONE JSON line (rank 0): elements/s of the whole job, GB/s and the
roofline fraction of the dominant kernel, the oracle's CPU throughput on a
bounded sample, an end-to-end number through host buffers, and the SM
clocks seen during the timed region.  With the default workload and one
GPU the line also carries, under "configs", the same measurements of every
other configuration: BERT-base 1-bit Adam, BERT-large 1-bit LAMB, the flat
2^20 case, the INT8 quantizer at 2^30 and the largest flat sweep point that
fits in memory.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload gpt-1.3b|bert-base|flat-1m|bert-large|int8|flat|
                              resnet50-mixed] [--no-extras]

N > 1 runs under torchrun as independent replicas (one per GPU, no
collective on the data path); timing is the max over ranks.
--impl reference times the oracle (plain single-threaded C++) on the host
cores, on a bounded sample of the same workload.
"""
import argparse
import ctypes as ct
import hashlib
import json
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = ("fused 1-bit compress+update elements/s and HBM GB/s (% of roofline) at 1 GPU")
NOMINAL_HBM_GBS = 8000.0


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ---------------------------------------------------------------------------
# Algorithmic bytes per real element (G = gradient bytes, W workers)
# ---------------------------------------------------------------------------

def bytes_per_element(W, G, lamb=False, sign_m=False):
    """compress: m read 4 (sign form: the server's word, 1/8, once per group
    of up to 4 workers for Adam -- 2 with bf16 gradients -- once per tile for
    LAMB) + per worker
    g read G, e read 4 + write 4, old sign word read 1/8 + new word write
    1/8; server: W/8 word reads, e_s read 4 + write 4, sign word 1/8 + 1/8;
    Adam: sign word 1/8, v 4, p 4 + 4, m write 4 (none in sign form).  LAMB
    pass A: sign word 1/8, m 4+4, v_fresh 4+4, v_Tw 4; pass B: m 4, v_Tw 4,
    p 4+4.  LAMB in sign form: pass A reads the previous and the current
    sign word (1/8 + 1/8) instead of m, pass B the current word instead of
    m, and m is not written."""
    grp = 2 if G == 2 else 4
    comp = (0.125 * (1 if lamb else (W + grp - 1) // grp) if sign_m else 4) + W * (G + 8 + 0.25)
    serv = W / 8 + 8 + 0.25
    if lamb:
        upd = (0.25 + 12 + 0.125 + 12) if sign_m else (0.125 + 20 + 16)
    else:
        upd = 0.125 + 4 + 8 + (0 if sign_m else 4)
    return {"compress": comp, "server": serv, "update": upd, "total": comp + serv + upd}


# ---------------------------------------------------------------------------
# Clock sampling (NVML through ctypes; falls back to nvidia-smi)
# ---------------------------------------------------------------------------

REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
           0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
           0x2: "applications_clocks_setting", 0x1: "gpu_idle"}


class ClockSampler:
    """Samples the SM clock and the clock-event reasons of one GPU every
    ~2 ms in a thread while active (reads only; changes no setting)."""

    def __init__(self, uuid):
        self.samples = []
        self.max_mhz = None
        self._stop = threading.Event()
        self._t = None
        self._nvml = None
        self._h = None
        try:
            nv = ct.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit")
            h = ct.c_void_p()
            if nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ct.byref(h)) != 0:
                if nv.nvmlDeviceGetHandleByIndex_v2(0, ct.byref(h)) != 0:
                    raise OSError("nvml handle")
            mx = ct.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ct.byref(mx)) == 0:
                self.max_mhz = mx.value
            self._nvml, self._h = nv, h
            fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None)
            self._reasons_fn = fn or nv.nvmlDeviceGetCurrentClocksThrottleReasons
        except (OSError, AttributeError) as e:
            log(f"[bench] NVML unavailable ({e}); clocks via nvidia-smi")

    def _run(self):
        nv, h = self._nvml, self._h
        mhz, rs = ct.c_uint(), ct.c_ulonglong()
        while not self._stop.is_set():
            if nv.nvmlDeviceGetClockInfo(h, 1, ct.byref(mhz)) == 0:
                r = rs.value if self._reasons_fn(h, ct.byref(rs)) == 0 else 0
                self.samples.append((mhz.value, r))
            time.sleep(0.002)

    def _run_smi(self):
        import subprocess
        q = "clocks.sm,clocks.max.sm,clocks_event_reasons.active"
        while not self._stop.is_set():
            try:
                out = subprocess.run(["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits"],
                                     capture_output=True, text=True, timeout=5).stdout
                a = out.strip().splitlines()[0].split(",")
                self.max_mhz = int(float(a[1]))
                self.samples.append((int(float(a[0])), int(a[2].strip(), 16)))
            except Exception:
                pass
            time.sleep(0.05)

    def __enter__(self):
        self._t = threading.Thread(target=self._run if self._nvml else self._run_smi, daemon=True)
        self._t.start()
        return self

    def __exit__(self, *a):
        self._stop.set()
        self._t.join()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0}
        mhz = [s for s, _ in self.samples]
        bits = 0
        for _, r in self.samples:
            bits |= r
        names = [v for k, v in sorted(REASONS.items()) if bits & k and v != "gpu_idle"]
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": self.max_mhz,
                "reasons": names, "samples": len(self.samples)}


# ---------------------------------------------------------------------------
# Device-side synthetic inputs (same recipe as synth: per-tensor std
# 1e-3 * 10^U(-1, 1), Gaussian values; drawn on the GPU for speed)
# ---------------------------------------------------------------------------

def device_grads(torch, wl, n_pad, step, dtype, device):
    std = torch.zeros(n_pad, dtype=torch.float32, device=device)
    if wl.tensors is None:
        std[: wl.n] = wl.flat_std
    else:
        sizes = torch.tensor([s for _, s, _ in wl.tensors], device=device)
        std[: wl.n] = torch.repeat_interleave(
            torch.tensor(wl.layer_std, dtype=torch.float32, device=device), sizes)
    out = []
    for w in range(wl.W):
        gen = torch.Generator(device=device)
        gen.manual_seed(synth.SEED_BASE + 1000 * step + w)
        g = torch.randn(n_pad, generator=gen, device=device, dtype=torch.float32) * std
        out.append(g.to(dtype))
    return out


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def kernel_source_hash(files=("k_compress.cu", "ob_internal.cuh")):
    """Hash of the kernel sources a recorded measurement was taken on, with
    comments and blank space left out (they do not change the kernel)."""
    import re
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "momentum_compression_gb300", "csrc", f)) as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


INT8_SOURCES = ("k_int8.cu", "sround.cuh", "philox.cuh", "ob_internal.cuh")



def issue_threads_per_clk(props):
    """Issue rate of the GPU in thread instructions per clock: its SMs x 4
    schedulers x one warp instruction (32 thread instructions) per clock."""
    return props.multi_processor_count * 4 * 32


def recorded_kv(name, source_files):
    """key: value lines of a committed ncu summary under profiles/, if it was
    taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", name)
    try:
        kv = {}
        for line in open(path):
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
        if kv.get("source_hash") != kernel_source_hash(source_files):
            return None
        return kv
    except OSError:
        return None


def recorded_traffic(workload, sign_m):
    """DRAM bytes per element of the compress kernel from the committed ncu
    summary (profiles/compress_traffic.txt), if it was taken on the current
    kernel source and on the same kernel variant: the worker count, the
    gradient type, the momentum's form and the mode.  The capture is made on
    a small case of that variant (a few GB on the device) and the bytes per
    element carry over to any size: the kernel streams every array once,
    with no reuse the L2 could change."""
    path = os.path.join(ROOT, "profiles", "compress_traffic.txt")
    try:
        kv = {}
        for line in open(path):
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
        if kv.get("source_hash") != kernel_source_hash():
            return None
        if kv.get("workload_W") != str(workload.W) or kv.get("grad_bytes") != (
                "2" if workload.grad_dtype == "bf16" else "4"):
            return None
        if kv.get("momentum") != ("sign" if sign_m else "dense") or \
                kv.get("mode", "adam") != workload.mode:
            return None
        return float(kv["dram_bytes_per_element"])
    except (OSError, KeyError, ValueError):
        return None


# ---------------------------------------------------------------------------
# CPU baseline: the oracle, single-threaded, on a bounded sample
# ---------------------------------------------------------------------------

def oracle_sample_step_time(wl, sample, steps, budget_s=None):
    """Per-step times of the oracle's compressed step (1-bit Adam, or 1-bit
    LAMB for a LAMB workload) on the first `sample` elements of the
    workload: `steps` steps, or with budget_s, steps until budget_s seconds
    have passed (at least 2, at most `steps`)."""
    import oracle as O
    lamb = wl.mode == "lamb"
    lay = O.Layout(sample, wl.W, wl.align, wl.chunk)
    layers = None
    if lamb:  # the workload's layers cut at the sample's end
        offs = [int(o) for o in (wl.layer_offsets if wl.layer_offsets is not None else [0])
                if int(o) < sample] + [sample]
        layers = O.Layers(np.array(offs, np.uint64))
    st = O.State(lay, layers, lamb=lamb)
    st.v[:sample] = synth.state_slice(wl, "v", 0, sample)
    st.m[:sample] = synth.state_slice(wl, "m", 0, sample)
    if lamb:  # compressed-phase LAMB state drawn directly: sigma = c = r = 1
        st.v_fresh[:] = st.v
        L = layers.count()
        st.ls = {k: np.ones(L, np.float32) for k in ("s", "c_avg", "r_prev", "c_prev", "c_prev2")}
    grads = []
    for w in range(wl.W):
        a = np.zeros(lay.n_pad, np.float32)
        a[:sample] = synth.grad_slice(wl, 0, w, 0, sample)
        if wl.grad_dtype == "bf16":
            a = synth.bf16_to_f32(synth.bf16_bits(a))
        grads.append(a)
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        O.compressed_step(st, grads, wl.hp, lamb=lamb)
        times.append(time.perf_counter() - t0)
        if budget_s is not None and len(times) >= 2 and sum(times) >= budget_s:
            break
    return times


def cpu_model():
    import platform
    import subprocess
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return f"{line.split(':', 1)[1].strip()} ({platform.machine()})"
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.machine()


# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x, dist=None, device="cpu"):
    """The largest value of x over all ranks (x itself without a process
    group).  Timing takes the max: the job is as slow as its slowest rank."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank, world, ms):
    """Units per second of the whole job: every rank processes
    units_per_rank, the job takes ms (max over ranks)."""
    return world * units_per_rank / (ms * 1e-3)


def run_reference(args, wl):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    sample = min(1 << 21, wl.n)
    steps = max(args.steps, 1)
    times = oracle_sample_step_time(wl, sample, args.warmup + steps)[args.warmup:]
    t = sum(times) / len(times)
    value = sample / t
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "elements/s",
        "n_gpus": args.gpus, "steps": steps, "warmup": args.warmup, "ms_per_step": t * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": f"{wl.name} (oracle on a {sample}-element sample)", "n": wl.n,
                   "W": wl.W, "chunk": wl.chunk, "parallelism": "replicas"},
        "cpu_baseline": {"value": value, "unit": "elements/s", "cores": 1, "kind": "oracle",
                         "sample": f"first {sample} elements of {wl.name}, W={wl.W}, "
                                   f"one compressed step per timed step", "cpu": cpu_model()},
        "e2e": {"value": value, "unit": "elements/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_int8(args, n=None, ef=None):
    """The block-256 INT8 stochastic-rounding quantizer on the sweep's
    largest size, n = 2^30 fp32 values (4 GB in, 1 GB of codes and 16 MB of
    scales out per call; larger than L2).  ef (--ef): with error feedback
    (the residual is read and written, 13 B per element) and the per-block
    error monitor.  Returns the JSON line (rank 0) or None."""
    import torch

    import momentum_compression_gb300 as ob
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    n = n or args.n or (1 << 30)
    ef = args.ef if ef is None else ef
    g = torch.randn(n, device="cuda") * 1e-3
    q = torch.empty(n, dtype=torch.int8, device="cuda")
    sc = torch.empty((n + 255) // 256, device="cuda")
    e = torch.zeros(n, device="cuda") if ef else None
    e2 = torch.empty((n + 255) // 256, device="cuda") if ef else None

    def call(t):
        if ef:
            ob.ob_quant_int8_ef(g, e, q, sc, 1234, t, None, e2)
        else:
            ob.ob_quant_int8(g, q, sc, 1234, t)

    for t in range(args.warmup):
        call(t)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    props = torch.cuda.get_device_properties(local)
    uuid = getattr(props, "uuid", None)
    uuid = f"GPU-{uuid}" if uuid is not None and not str(uuid).startswith("GPU-") else str(uuid)
    with ClockSampler(uuid) as clk:
        torch.cuda.synchronize()
        a.record(stream)
        for t in range(args.steps):
            call(1000 + t)
        b.record(stream)
        torch.cuda.synchronize()
    ms = a.elapsed_time(b) / args.steps
    bpe = (4 + 4 + 4 + 1 + 8 / 256) if ef else (4 + 1 + 4 / 256)
    peak, kind = measured_peak()
    gbs = bpe * n / (ms * 1e-3) / 1e9
    clocks = clk.summary()
    # The quantizer is bound by instruction issue, not by HBM: its roofline
    # is the issue rate at the clock seen, against the thread instructions
    # per element that ncu counted for this kernel source (profiles/).
    kv = recorded_kv("int8_instructions.txt", INT8_SOURCES) or {}
    ipe = kv.get("thread_instructions_per_element_ef" if ef else
                 "thread_instructions_per_element")
    mhz = clocks.get("sm_mhz") or clocks.get("sm_max_mhz") or 2070
    issue_peak = issue_threads_per_clk(props) * mhz * 1e6 / 1e12
    if ipe is not None:
        ach = float(ipe) * n / (ms * 1e-3) / 1e12
        roofline = {"bound": "alu", "kernel": "quant_int8", "achieved": ach,
                    "peak": issue_peak, "peak_kind": f"issue rate at the median SM clock "
                    f"({mhz:.0f} MHz): {props.multi_processor_count} SMs x 4 schedulers x 32 "
                    "lanes",
                    "unit": "T thread-instructions/s", "frac": ach / issue_peak,
                    "instructions_per_element": float(ipe),
                    "hbm": {"achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                            "bytes_per_element": bpe}, "traffic": None}
    else:
        roofline = {"bound": "hbm", "kernel": "quant_int8", "achieved": gbs, "peak": peak,
                    "peak_kind": kind, "unit": "GB/s", "frac": gbs / peak,
                    "bytes_per_element": bpe, "traffic": None,
                    "note": "no instruction count recorded for this kernel source"}
    if rank == 0:
        what = "with error feedback and error monitor" if ef else ""
        return {
            "metric": "INT8 block-256 stochastic-rounding quantizer elements/s", "value": n / (ms * 1e-3),
            "unit": "elements/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32 -> int8", "data": "synthetic",
            "config": {"workload": f"int8 quantizer {what}, n = {n}, block 256, Philox4x32-10",
                       "l2": "inputs larger than L2; no flush"},
            "roofline": roofline, "gpu_launches": args.steps, "clocks": clocks}
    return None


def run_ours(args, wl, with_e2e=True, with_cpu=True, grad_sets=2):
    """One 1-bit workload: warmup steps, then K timed compressed steps
    (eager with per-kernel events, and CUDA-graph replays), the end-to-end
    step through host buffers (with_e2e) and the oracle's CPU rate on a
    bounded sample (with_cpu).  grad_sets: resident gradient sets the steps
    alternate between (1 for the largest sweep point, whose memory it
    saves).  Returns the JSON line (rank 0) or None."""
    import torch

    import momentum_compression_gb300 as ob

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
        pg = dist
    G = 2 if wl.grad_dtype == "bf16" else 4
    gdt = torch.bfloat16 if wl.grad_dtype == "bf16" else torch.float32
    sign_m = not args.dense_m
    opt = ob.OneBitOptimizer(wl.n, wl.W, wl.chunk, wl.align, wl.grad_dtype, wl.layer_offsets,
                             lamb=(wl.mode == "lamb"), device=device, sign_momentum=sign_m,
                             **wl.hp)
    n, n_pad = wl.n, opt.n_pad
    log(f"[bench] rank {rank}: {wl.name} n={n} W={wl.W} n_pad={n_pad} "
        f"tiles={opt.layout['n_tiles']}")
    # parameters and two resident gradient sets
    p0 = torch.zeros(n_pad, device=device)
    gen = torch.Generator(device=device)
    gen.manual_seed(synth.SEED_BASE + 17)
    p0[:n] = torch.randn(n, generator=gen, device=device) * 0.02
    opt.p.copy_(p0)
    del p0
    gsets = [device_grads(torch, wl, n_pad, s, gdt, device) for s in range(grad_sets)]
    if grad_sets == 1:
        gsets = gsets * 2
    # prerequisite: a few uncompressed warmup steps freeze v (timed on their
    # own: the warmup step is a row of the path, not the metric)
    stream0 = torch.cuda.current_stream()
    wa, wb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    opt.warmup_step(gsets[0])
    wa.record(stream0)
    for t in range(1, 4):
        opt.warmup_step(gsets[t % 2])
    wb.record(stream0)
    torch.cuda.synchronize()
    warm_ms = wa.elapsed_time(wb) / 3
    opt.begin_compression()
    stream = torch.cuda.current_stream()
    for t in range(args.warmup):
        opt.compressed_step(gsets[t % 2])
    torch.cuda.synchronize()
    if sign_m and not opt.m_in_signs:
        raise SystemExit("bench: the sign-form momentum starts after one compressed step; "
                         "give --warmup >= 1")

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    props = torch.cuda.get_device_properties(device)
    uuid = getattr(props, "uuid", None)
    uuid = f"GPU-{uuid}" if uuid is not None and not str(uuid).startswith("GPU-") else str(uuid)
    lamb = opt.lamb
    db = opt.double_buffered  # LAMB in sign form: two server buffers

    # the three rows of a compressed step through the public calls
    def compress(g):
        if db:
            ob.ob_compress_signm_ls(opt.ctx, g, opt.sbits, opt.sscales, opt.err, opt.bits,
                                    opt.scales, opt.ls)
        elif sign_m:
            ob.ob_compress_signm(opt.ctx, g, opt.sbits, opt.sscales, opt.err, opt.bits,
                                 opt.scales)
        else:
            ob.ob_compress(opt.ctx, g, opt.m, opt.err, opt.bits, opt.scales, opt.ls)

    def server():
        if db:
            ob.ob_server_reduce_db(opt.ctx, opt.bits, opt.scales, opt.err_s, opt.sbits,
                                   opt.sscales, opt.sbits_alt, opt.sscales_alt, opt.ls)
        else:
            ob.ob_server_reduce(opt.ctx, opt.bits, opt.scales, opt.err_s, opt.sbits, opt.sscales,
                                opt.ls)

    def update():
        if db:
            ob.ob_lamb_step_signm(opt.ctx, opt.sbits, opt.sscales, opt.sbits_alt,
                                  opt.sscales_alt, opt.v, opt.v_fresh, opt.p, opt.ls)
            opt._swap()  # this step's output becomes the current pair
        elif lamb:
            ob.ob_lamb_step(opt.ctx, opt.sbits, opt.sscales, opt.v, opt.v_fresh, opt.m, opt.p,
                            opt.ls)
        else:
            ob.ob_adam_step(opt.ctx, opt.sbits, opt.sscales, opt.v, None if sign_m else opt.m,
                            opt.p)

    with ClockSampler(uuid) as clk:
        if pg:
            pg.barrier()
        torch.cuda.synchronize()
        t_start.record(stream)
        for t in range(K):
            g = gsets[t % 2]
            e = ev[t]
            e[0].record(stream)
            compress(g)
            e[1].record(stream)
            server()
            e[2].record(stream)
            update()
            e[3].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
        if pg:
            pg.barrier()
    total_ms = t_start.elapsed_time(t_end)
    per = {k: [ev[t][i].elapsed_time(ev[t][i + 1]) for t in range(K)]
           for i, k in enumerate(("compress", "server", "update"))}
    graph_info = None
    clocks = clk.summary()
    if not args.eager:
        # The same steps replayed from CUDA graphs (one per gradient set,
        # OneBitOptimizer.capture_step): one launch per step instead of five
        # or six.  Per-kernel times come from the eager loop above; the step
        # time, and the clocks reported with it, from the replays.
        graphs = [opt.capture_step(gsets[i]) for i in range(2)]
        for t in range(2):
            graphs[t % 2].replay()
        torch.cuda.synchronize()
        ga, gb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(uuid) as gclk:
            if pg:
                pg.barrier()
            torch.cuda.synchronize()
            ga.record(stream)
            for t in range(K):
                graphs[t % 2].replay()
            gb.record(stream)
            torch.cuda.synchronize()
            if pg:
                pg.barrier()
        eager_ms = max_over_ranks(total_ms, pg, device) / K
        total_ms = ga.elapsed_time(gb)
        graph_info = {"eager_ms_per_step": eager_ms, "graph_launches_per_step": 1,
                      "eager_clocks": clocks}
        clocks = gclk.summary()
        del graphs
    # compress + scale finalisation, server + scale finalisation, update
    # (LAMB: pass A and pass B); the kernels inside a replayed graph count too
    launches = K * (6 if lamb else 5)
    total_ms = max_over_ranks(total_ms, pg, device)
    ms = total_ms / K
    bpe = bytes_per_element(wl.W, G, lamb, sign_m)
    # warmup: W gradients read; m, v, p read + written (LAMB: pass 1 reads
    # g, m, v, p and writes m, v; pass 2 reads m, v, p and writes p)
    warm_bpe = wl.W * G + (36 if lamb else 24)
    value = job_rate(n, world, ms)
    peak, peak_kind = measured_peak()
    kms = {k: sum(v) / K for k, v in per.items()}
    dom = max(kms, key=kms.get)
    dom_bytes = bpe[dom] * n
    achieved = dom_bytes / (kms[dom] * 1e-3) / 1e9
    traffic = recorded_traffic(wl, sign_m) if dom == "compress" else None

    e2e = None
    if with_e2e:
        # End to end through host buffers, pipelined through the public calls.
        # Every step copies all W gradients host -> device (pinned memory) and
        # reads the updated parameters back.  A copy stream brings step t+1's
        # gradients into the other device buffer set while the compute stream
        # runs step t; a read-back stream copies step t's parameters to the
        # host, and the update of step t+1 waits for that read-back (it
        # rewrites p).  The host link (about 210 GB/s here) bounds it.
        host_g = [torch.empty(n_pad, dtype=gdt, pin_memory=True) for _ in range(wl.W)]
        for w in range(wl.W):
            host_g[w].copy_(gsets[0][w])
        host_p = torch.empty(n_pad, dtype=torch.float32, pin_memory=True)
        s_h2d, s_d2h = torch.cuda.Stream(device), torch.cuda.Stream(device)
        ev = lambda: torch.cuda.Event()
        ev_h2d, ev_used = [ev(), ev()], [ev(), ev()]
        ev_upd, ev_back = ev(), ev()

        def issue_h2d(t):
            b = t % 2
            if t >= 2:
                s_h2d.wait_event(ev_used[b])
            with torch.cuda.stream(s_h2d):
                for w in range(wl.W):
                    gsets[b][w].copy_(host_g[w], non_blocking=True)
            ev_h2d[b].record(s_h2d)

        def issue_step(t):
            b = t % 2
            stream.wait_event(ev_h2d[b])
            compress(gsets[b])
            server()
            ev_used[b].record(stream)
            if t >= 1:
                stream.wait_event(ev_back)
            update()
            ev_upd.record(stream)
            s_d2h.wait_event(ev_upd)
            with torch.cuda.stream(s_d2h):
                host_p.copy_(opt.p, non_blocking=True)
            ev_back.record(s_d2h)

        def pipeline(steps):
            issue_h2d(0)
            for t in range(steps):
                if t + 1 < steps:
                    issue_h2d(t + 1)
                issue_step(t)

        pipeline(2)
        torch.cuda.synchronize()
        K2 = max(3, min(K, 10))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s_h2d)
        pipeline(K2)
        b.record(s_d2h)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(a.elapsed_time(b) / K2, pg, device)
        e2e = {"value": job_rate(n, world, e2e_ms), "unit": "elements/s",
               "h2d_bytes_per_step": wl.W * n_pad * G, "d2h_bytes_per_step": n_pad * 4,
               "ms_per_step": e2e_ms,
               "pipelined": "H2D of step t+1 overlaps step t and its parameter read-back"}
        del host_g, host_p

    cpu = None
    if with_cpu and rank == 0 and world == 1:
        sample = min(1 << 24, n)
        times = oracle_sample_step_time(wl, sample, 16, budget_s=12.0)
        steps = len(times)
        cpu = {"value": sample * steps / sum(times), "unit": "elements/s", "cores": 1,
               "kind": "oracle",
               "sample": f"first {sample} elements of {wl.name}, W={wl.W}, {steps} compressed "
                         f"{'1-bit LAMB' if wl.mode == 'lamb' else '1-bit Adam'} steps "
                         f"({sum(times):.1f} s)", "cpu": cpu_model()}

    if rank != 0:
        opt.close()
        return None
    line = {
        "metric": METRIC, "value": value, "unit": "elements/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32" if G == 4 else "f32 (bf16 gradients)",
        "data": "synthetic",
        "config": {"workload": wl_label(wl), "n": n, "W": wl.W, "chunk": wl.chunk,
                   "momentum": (("sign form, server output double-buffered, exact "
                                 "(ob_compress_signm_ls, ob_lamb_step_signm)") if db else
                                "sign form: sbits + chunk scales, exact (ob_compress_signm)"
                                if sign_m else "dense fp32"),
                   "n_layers": wl.n_layers, "grad_dtype": wl.grad_dtype,
                   "parallelism": "replicas" if world > 1 else "1 GPU",
                   "l2": f"inputs larger than L2 ({bpe['total'] * n / 1e9:.1f} GB touched per "
                         f"step); no flush"},
        "gbs": bpe["total"] * n / (ms * 1e-3) / 1e9,
        "worker_elements_per_s": world * n * wl.W / (ms * 1e-3),
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                     "frac_of_nominal_8000": achieved / NOMINAL_HBM_GBS,
                     "bytes_per_element": bpe[dom],
                     "traffic": None if traffic is None else traffic * n},
        "step_roofline_frac": bpe["total"] * n / (ms * 1e-3) / 1e9 / peak,
        "warmup_step": {"ms": warm_ms, "bytes_per_element": warm_bpe,
                        "gbs": warm_bpe * n / (warm_ms * 1e-3) / 1e9},
        "kernels_ms": kms,
        "kernels_gbs": {k: bpe[k] * n / (kms[k] * 1e-3) / 1e9 for k in kms},
        "gpu_launches": launches,
        "clocks": clocks,
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    if graph_info is not None:
        line["config"]["launch"] = "CUDA graph replay (one graph launch per step)"
        line["graph"] = graph_info
    opt.close()
    return line


def mixed_bytes(bits, W, G, send=True):
    """Algorithmic bytes per real element of one mixed-width group, per
    kernel: b-bit codes are b/8 bytes per element plus a 4-byte scale per
    256; FP16 messages are 2 bytes, exchanged on sending steps only."""
    if bits == 16:
        comp = 4 + W * (G + 8 + (2 if send else 0))
        serv = (W * 2 + 8 + 2) if send else 0
        upd = (2 + 4 + 8 + 4) if send else 4
    else:
        code = bits / 8 + 4 / 256
        comp = 4 + W * (G + 8 + code)
        serv = W * code + 8 + code
        upd = code + 4 + 8 + 4
    return {"compress": comp, "server": serv, "update": upd, "total": comp + serv + upd}


def run_mixed(args):
    """Layerwise mixed bit widths on the ResNet-50 parameter list: 1-bit
    scaled sign for the fc layer, the 2-bit block codec for the
    convolutions, FP16 every 10th step for the batch-norm parameters, W = 8.
    One step = one compressed step of every group."""
    import torch

    import momentum_compression_gb300 as ob
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
        pg = dist
    groups = synth.mixed_groups(W=args.W or 8)
    W = groups[0][1].W
    sign_m = not args.dense_m
    specs = [(bits, wl.n, wl.layer_offsets) for bits, wl in groups]
    opt = ob.MixedOptimizer(specs, W, chunk=1 << 20, period=synth.NORM_PERIOD, seed=1234,
                            device=device, sign_momentum=sign_m, **synth.ADAM_HP)
    n_tot = sum(wl.n for _, wl in groups)
    log(f"[bench] rank {rank}: resnet50-mixed n={n_tot} W={W} groups "
        + ", ".join(f"{b}-bit {wl.n}" for b, wl in groups))
    gsets = [[device_grads(torch, wl, g.n_pad, s, torch.float32, device)
              for (_, wl), (_, g) in zip(groups, opt.groups)] for s in range(2)]
    for _, g in opt.groups:
        g.p.normal_(0.0, 0.02)
    for t in range(3):
        opt.warmup_step(gsets[t % 2])
    opt.begin_compression()
    for t in range(args.warmup):
        opt.compressed_step(gsets[t % 2])
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    K = args.steps
    ng = len(groups)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(ng + 1)] for _ in range(K)]
    kev = {}  # per-kernel events of the 2-bit group's step
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    props = torch.cuda.get_device_properties(device)
    uuid = getattr(props, "uuid", None)
    uuid = f"GPU-{uuid}" if uuid is not None and not str(uuid).startswith("GPU-") else str(uuid)
    sends = 0
    with ClockSampler(uuid) as clk:
        if pg:
            pg.barrier()
        torch.cuda.synchronize()
        t_start.record(stream)
        for t in range(K):
            e = ev[t]
            e[0].record(stream)
            for i, ((bits, _), (_, g)) in enumerate(zip(groups, opt.groups)):
                if bits == 2:
                    # the group's three calls, with an event between each
                    ke = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
                    g.t += 1
                    ob.ob_compress_qb(g.ctx, 2, gsets[t % 2][i], g.m, g.err, g.codes, g.bscales,
                                      g.key, g.t)
                    ke[0].record(stream)
                    ob.ob_server_reduce_qb(g.ctx, 2, g.codes, g.bscales, g.err_s, g.scodes,
                                           g.sbscales, g.key, g.t)
                    ke[1].record(stream)
                    ob.ob_adam_step_qb(g.ctx, 2, g.scodes, g.sbscales, g.v, g.m, g.p)
                    ke[2].record(stream)
                    kev[t] = (e[i], ke)
                else:
                    if bits == 16 and (g.t + 1) % g.period == 0:
                        sends += 1
                    g.compressed_step(gsets[t % 2][i])
                e[i + 1].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
        if pg:
            pg.barrier()
    total_ms = max_over_ranks(t_start.elapsed_time(t_end), pg, device)
    ms = total_ms / K
    group_ms = {f"{bits}-bit": sum(ev[t][i].elapsed_time(ev[t][i + 1]) for t in range(K)) / K
                for i, (bits, _) in enumerate(groups)}
    kq = {}
    for name, j in (("compress", 0), ("server", 1), ("update", 2)):
        kq[name] = sum((kev[t][0] if j == 0 else kev[t][1][j - 1]).elapsed_time(kev[t][1][j])
                       for t in range(K)) / K
    nq = dict(groups)[2].n
    bq = mixed_bytes(2, W, 4)
    kq_gbs = {k: bq[k] * nq / (kq[k] * 1e-3) / 1e9 for k in kq}
    launches = K * (5 + 3 + 2) + sends
    peak, peak_kind = measured_peak()
    frac_send = sends / K
    total_bytes = 0.0
    for bits, wl in groups:
        if bits == 1:
            total_bytes += bytes_per_element(W, 4, False, sign_m)["total"] * wl.n
        elif bits == 16:
            total_bytes += (frac_send * mixed_bytes(16, W, 4, True)["total"] +
                            (1 - frac_send) * mixed_bytes(16, W, 4, False)["total"]) * wl.n
        else:
            total_bytes += mixed_bytes(bits, W, 4)["total"] * wl.n

    # end to end through host buffers: every step copies all groups' W
    # gradients host -> device from pinned memory, runs the step and reads
    # all parameters back, in order on one stream
    host_g = [[torch.empty_like(x, device="cpu").pin_memory() for x in gs] for gs in gsets[0]]
    for hg, dg in zip(host_g, gsets[0]):
        for h, d in zip(hg, dg):
            h.copy_(d)
    host_p = [torch.empty(g.n_pad, pin_memory=True) for _, g in opt.groups]

    def e2e_step(t):
        for hg, dg in zip(host_g, gsets[t % 2]):
            for h, d in zip(hg, dg):
                d.copy_(h, non_blocking=True)
        opt.compressed_step(gsets[t % 2])
        for hp_, (_, g) in zip(host_p, opt.groups):
            hp_.copy_(g.p, non_blocking=True)

    e2e_step(0)
    torch.cuda.synchronize()
    K2 = max(3, min(K, 10))
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for t in range(K2):
        e2e_step(t)
    b.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(a.elapsed_time(b) / K2, pg, device)
    h2d = sum(x.numel() * x.element_size() for hg in host_g for x in hg)
    d2h = sum(x.numel() * 4 for x in host_p)
    e2e = {"value": job_rate(n_tot, world, e2e_ms), "unit": "elements/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
           "pipelined": False}
    del host_g, host_p

    cpu = None
    if rank == 0 and world == 1:
        cpu = mixed_oracle_sample(groups, steps=3)
    if rank != 0:
        opt.close()
        return
    achieved = kq_gbs["compress"]
    line = {
        "metric": "layerwise mixed-width compressed step elements/s (1-bit / 2-bit / FP16 "
                  "groups)", "value": job_rate(n_tot, world, ms), "unit": "elements/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": "resnet50-mixed: ResNet-50 parameter list (161 tensors, "
                               f"{n_tot:,} params), W={W}; fc 1-bit, convolutions 2-bit "
                               "(block 256), batch norms FP16 every 10th step",
                   "groups": {f"{b}-bit": wl.n for b, wl in groups}, "W": W,
                   "momentum_1bit": "sign form" if sign_m else "dense fp32",
                   "parallelism": "replicas" if world > 1 else "1 GPU",
                   "l2": f"inputs larger than L2 ({total_bytes / 1e9:.1f} GB touched per step);"
                         " no flush"},
        "gbs": total_bytes / (ms * 1e-3) / 1e9,
        "group_ms": group_ms,
        "kernels_ms_2bit": kq, "kernels_gbs_2bit": kq_gbs,
        "roofline": {"bound": "hbm", "kernel": "qb_compress (2-bit group)", "achieved": achieved,
                     "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": achieved / peak, "bytes_per_element": bq["compress"],
                     "traffic": None},
        "step_roofline_frac": total_bytes / (ms * 1e-3) / 1e9 / peak,
        "gpu_launches": launches, "clocks": clk.summary(), "e2e": e2e, "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    opt.close()


def mixed_oracle_sample(groups, steps):
    """The oracle's mixed step on a bounded sample: the first 2^22 elements
    of each group (all of a smaller one), W workers, `steps` compressed
    steps; elements/s over the sampled elements."""
    import oracle as O
    total, t_all, names = 0, 0.0, []
    for bits, wl in groups:
        sample = min(1 << 22, wl.n)
        lay = O.Layout(sample, wl.W, wl.align, wl.chunk)
        st = O.State(lay)
        st.v[:sample] = synth.state_slice(wl, "v", 0, sample)
        st.m[:sample] = synth.state_slice(wl, "m", 0, sample)
        grads = []
        for w in range(wl.W):
            a = np.zeros(lay.n_pad, np.float32)
            a[:sample] = synth.grad_slice(wl, 0, w, 0, sample)
            grads.append(a)
        t0 = time.perf_counter()
        for t in range(1, steps + 1):
            O.codec_step(st, grads, wl.hp, bits, t, 1234 + bits, period=synth.NORM_PERIOD)
        t_all += time.perf_counter() - t0
        total += sample * steps
        names.append(f"{sample} of the {bits}-bit group")
    return {"value": total / t_all, "unit": "elements/s", "cores": 1, "kind": "oracle",
            "sample": f"{', '.join(names)}, W={groups[0][1].W}, {steps} compressed steps "
                      f"({t_all:.1f} s)", "cpu": cpu_model()}


def run_sweep(args):
    """The flat bandwidth sweep: n in {2^20, 2^24, 2^28, 2^30} x W in {1, 2,
    4, 8, 16} x chunk in {2^12, 2^20} (chunk clamped to the partition),
    state drawn directly (m, e ~ N(0, 1e-3), v ~ |N(0, 1e-6)| + 1e-12, no
    warmup), 1-bit Adam with the momentum in sign form after the first
    step.  One JSON line per point: the step's elements/s and GB/s, and the
    compress kernel's GB/s.  Points that do not fit in free memory are
    skipped.  Small points are launch-bound and L2-resident."""
    import torch

    import momentum_compression_gb300 as ob
    torch.cuda.set_device(0)
    peak, kind = measured_peak()
    for n_log in (20, 24, 28, 30):
        for W in (1, 2, 4, 8, 16):
            for c_log in (12, 20):
                n, C = 1 << n_log, 1 << c_log
                need = n * (8 * W + 24) * 1.1
                free, _ = torch.cuda.mem_get_info()
                if need > free * 0.9:
                    log(f"[sweep] skip n=2^{n_log} W={W}: {need / 1e9:.0f} GB needed")
                    continue
                opt = ob.OneBitOptimizer(n, W, C, 4096, "f32", None, sign_momentum=True,
                                         **synth.ADAM_HP)
                gen = torch.Generator(device="cuda")
                gen.manual_seed(synth.SEED_BASE + n_log * 100 + W)
                opt.m[:n] = torch.randn(n, generator=gen, device="cuda") * 1e-3
                opt.v[:n] = torch.randn(n, generator=gen, device="cuda").abs() * 1e-6 + 1e-12
                for e in opt.err:
                    e[:n] = torch.randn(n, generator=gen, device="cuda") * 1e-3
                grads = [torch.zeros(opt.n_pad, device="cuda") for _ in range(W)]
                for g in grads:
                    g[:n] = torch.randn(n, generator=gen, device="cuda") * 1e-3
                K = 50 if n_log <= 24 else 10
                for _ in range(3):
                    opt.compressed_step(grads)
                torch.cuda.synchronize()
                stream = torch.cuda.current_stream()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                ca, cb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                for _ in range(K):
                    opt.compressed_step(grads)
                b.record(stream)
                ca.record(stream)
                for _ in range(K):
                    ob.ob_compress_signm(opt.ctx, grads, opt.sbits, opt.sscales, opt.err,
                                         opt.bits, opt.scales)
                cb.record(stream)
                torch.cuda.synchronize()
                ms = a.elapsed_time(b) / K
                cms = ca.elapsed_time(cb) / K
                bpe = bytes_per_element(W, 4, False, True)
                gbs = bpe["total"] * n / (ms * 1e-3) / 1e9
                cgbs = bpe["compress"] * n / (cms * 1e-3) / 1e9
                print(json.dumps({
                    "sweep": "flat 1-bit Adam, sign-form momentum", "n": n, "W": W,
                    "chunk": min(C, opt.layout["P"]), "steps": K, "ms_per_step": ms,
                    "elements_per_s": n / (ms * 1e-3), "gbs": gbs, "frac": gbs / peak,
                    "compress_ms": cms, "compress_gbs": cgbs, "compress_frac": cgbs / peak,
                    "peak": peak, "peak_kind": kind,
                    "l2": "L2-resident" if bpe["total"] * n < 2 * 129e6 else "larger than L2"}),
                    flush=True)
                opt.close()
                del grads, opt
                torch.cuda.empty_cache()


def wl_label(wl):
    kind = "1-bit LAMB" if wl.mode == "lamb" else "1-bit Adam"
    shape = f"{wl.n_layers} tensors" if wl.tensors else "flat"
    return (f"{wl.name} {kind}: {wl.n:,} params ({shape}) fused, W={wl.W} simulated workers, "
            f"chunk {wl.chunk}, {wl.grad_dtype} grads")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=("ours", "reference"))
    ap.add_argument("--workload", default=None,
                    help="default gpt-1.3b (the largest single-GPU configuration), with the "
                         "other configurations measured under \"configs\"")
    ap.add_argument("--n", "--elements", dest="n", type=int,
                    help="elements (flat and int8 workloads); use --elements under torchrun")
    ap.add_argument("--W", type=int, help="workers (flat workload only)")
    ap.add_argument("--chunk", type=int, help="chunk (flat workload only)")
    ap.add_argument("--grad-dtype", choices=("f32", "bf16"), default="f32",
                    help="gradient type (flat workload only)")
    ap.add_argument("--mode", choices=("adam", "lamb"), default="adam",
                    help="1-bit Adam or 1-bit LAMB (flat workload only; one layer)")
    ap.add_argument("--eager", action="store_true",
                    help="1-bit workloads: time the eager launches only (by default the step "
                         "is also captured in CUDA graphs and the replays are timed)")
    ap.add_argument("--graph", action="store_true",
                    help="kept for old command lines: graph replay is the default")
    ap.add_argument("--dense-m", action="store_true",
                    help="keep the momentum as a dense fp32 buffer (default: its exact sign form)")
    ap.add_argument("--ef", action="store_true", help="int8 workload: with error feedback")
    ap.add_argument("--clip-value", type=float, default=0.0,
                    help="clamp of the compensated values (the write-up's stability variant)")
    ap.add_argument("--sweep", action="store_true",
                    help="the flat n x W x chunk bandwidth sweep, one JSON line per point")
    ap.add_argument("--no-extras", action="store_true",
                    help="default workload: leave out the other configurations")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.sweep:
        run_sweep(args)
        return
    default = args.workload is None
    if default:
        args.workload = DEFAULT_WORKLOAD
    if args.impl == "ours" and args.workload == "int8":
        line = run_int8(args)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if args.workload == "resnet50-mixed":
        if args.impl == "reference":
            world, rank, _ = dist_env()
            if rank == 0:
                cpu = mixed_oracle_sample(synth.mixed_groups(), steps=min(max(args.steps, 1), 3))
                print(json.dumps({
                    "impl": "reference", "metric": "layerwise mixed-width compressed step "
                    "elements/s (1-bit / 2-bit / FP16 groups)", "value": cpu["value"],
                    "unit": "elements/s", "n_gpus": args.gpus, "steps": args.steps,
                    "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
                    "vs_baseline": None, "dtype": "f32", "data": "synthetic",
                    "config": {"workload": "resnet50-mixed (oracle on a sample)"},
                    "cpu_baseline": cpu,
                    "e2e": {"value": cpu["value"], "unit": "elements/s",
                            "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}), flush=True)
        else:
            run_mixed(args)
        return
    if args.workload == "flat":
        wl = synth.workload("flat", n=args.n or (1 << 24), W=args.W or 8,
                            chunk=args.chunk or (1 << 20), grad_dtype=args.grad_dtype)
        if args.mode == "lamb":
            wl.mode = "lamb"
            wl.hp.update(r_thr=0.1, r_min=0.5, r_max=4.0, c_min=0.01, c_max=10.0)
    else:
        wl = synth.workload(args.workload)
    if args.clip_value:
        wl.hp["clip_value"] = args.clip_value
    if args.impl == "reference":
        run_reference(args, wl)
        return
    line = run_ours(args, wl)
    world, rank, _ = dist_env()
    if default and world == 1 and not args.no_extras:
        line["configs"] = run_extras(args)
    if line is not None:
        print(json.dumps(line), flush=True)


DEFAULT_WORKLOAD = "gpt-1.3b"


def config_entry(line):
    """The measurements of one configuration as carried in the headline's
    "configs": its own step time, per-kernel times and GB/s, the roofline
    of its dominant kernel (bytes per element and kernel time, so the
    fraction recomputes), and the clocks seen while it ran."""
    keep = ("metric", "value", "unit", "ms_per_step", "steps", "dtype", "config", "gbs",
            "worker_elements_per_s", "roofline", "step_roofline_frac", "warmup_step",
            "kernels_ms", "kernels_gbs", "gpu_launches", "clocks", "graph")
    return {k: line[k] for k in keep if k in line}


def run_extras(args):
    """Every other configuration, one after the other on this GPU (N = 1),
    each with its buffers freed before the next: BERT-base 1-bit Adam,
    BERT-large 1-bit LAMB, the flat 2^20 case (launch-bound and
    L2-resident), the INT8 quantizer at 2^30, and the largest point of the
    flat sweep (n = 2^30, W = 16, chunk 2^20, or the largest W that fits)."""
    import gc

    import torch
    out = {}

    def settle():
        gc.collect()
        torch.cuda.synchronize()
        torch.cuda.empty_cache()

    for name in ("bert-base", "bert-large", "flat-1m"):
        settle()
        wl = synth.workload(name)
        log(f"[bench] extra configuration {name}")
        out[name] = config_entry(run_ours(args, wl, with_e2e=False, with_cpu=False))
    settle()
    log("[bench] extra configuration int8")
    out["int8-2^30"] = config_entry(run_int8(args, n=1 << 30, ef=False))
    settle()
    free, _ = torch.cuda.mem_get_info()
    for W in (16, 8, 4):
        n = 1 << 30
        # W gradient and error buffers, m, v, p, e_s, sign words: 8W + 20 B/element
        if n * (8 * W + 20) * 1.1 < free * 0.9:
            wl = synth.workload("flat", n=n, W=W, chunk=1 << 20)
            log(f"[bench] extra configuration flat 2^30 x {W}")
            out[f"flat-2^30-W{W}"] = config_entry(
                run_ours(args, wl, with_e2e=False, with_cpu=False, grad_sets=1))
            break
    settle()
    return out


if __name__ == "__main__":
    main()
