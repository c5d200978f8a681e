#!/usr/bin/env python
"""Benchmark of the 36-layer GPT-OSS-120B-shaped decode iteration on GB300.

One step = one decode iteration: 64 sequences (one new token each) through 36
layers that alternate sliding-window-128 and full attention over a KV cache of
8,192 positions, run as the two-stage intra-GPU spatial pipeline (stage A:
RMSNorm + QKV + attention; stage B: o-proj + router + SwiGLU experts +
combine) through the C ABI.  The same work run temporally (every kernel on all
SMs) is reported beside it.  Inputs are seeded synthetic tensors (random
weights of the per-GPU slice shape; no trained checkpoint) resident in HBM; the
working set (about 48 GB) is far larger than L2, so no flush is needed between
steps.

`python bench.py [--gpus N] [--steps K] [--warmup W]` prints one JSON line.
Under torchrun every rank runs an independent replica (the path has no
cross-GPU exchange) and rank 0 prints the aggregate.
`--impl reference` times the fp64 CPU oracle on a bounded sample instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "36-layer decode iteration µs, tokens/s/GPU; DRAM GB/s as % of HBM peak"
UNIT = "tokens/s"
CSRC = os.path.join(ROOT, "intra_spatial_pipelining_gb300", "csrc")
# the attention kernel's sources: its own file and the device helpers it includes
ATTN_SRCS = [os.path.join(CSRC, f) for f in ("k_attention.cu", "common.cuh", "kernels.h")]
TRAFFIC_SUMMARY = os.path.join(ROOT, "profiles", "attn_decode_kernel_gptoss_36l.md")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="sgp", choices=["sgp", "reference"])
    ap.add_argument("--workload", default="gptoss_36l")
    ap.add_argument("--layers", type=int, default=None, help="override the layer count")
    ap.add_argument("--kv-len", type=int, default=None, help="override the KV length")
    ap.add_argument("--stages", type=int, default=2)
    ap.add_argument("--micro", type=int, default=None, help="sequences per microbatch")
    ap.add_argument("--split", default="auto",
                    help="'auto' (balancer, checked on its 4 best picks), 'sweep' (every legal "
                         "split as a full run) or a comma list of SMs")
    ap.add_argument("--cut", default="auto", choices=["auto", "layer", "macro", "macro_qkv", "macro_oproj"],
                    help="macro: full-attention decode alone on stage A, everything else on B; "
                         "macro_qkv: also the full layers' RMSNorm-1 and QKV projection on A; "
                         "macro_oproj: the full layers' ops up to the output projection on A; "
                         "layer: ops 0-2 of every layer on A; auto: the faster of macro and "
                         "macro_qkv after each one's split search")
    ap.add_argument("--no-temporal", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--virtual-comm", action="store_true",
                    help="add the pages' virtual communication kernels (3 us + bytes / 900 GB/s "
                         "for the attention all-reduce, MoE dispatch and MoE combine)")
    ap.add_argument("--lanes", type=int, default=2, choices=[1, 2],
                    help="FIFOs per stage: 1 = the pages' model, 2 = one per microbatch parity "
                         "(two streams per SM pool, as the pages' prototype runs)")
    ap.add_argument("--weight-reuse", action="store_true",
                    help="load the weights of every microbatch but the last with an L2 "
                         "evict-last hint (sgp_pipeline_opts.weight_reuse)")
    ap.add_argument("--no-paper-shape", action="store_true",
                    help="skip the secondary measurement at the pages' own decode shape")
    ap.add_argument("--frontier", action="store_true",
                    help="per-user vs per-GPU throughput frontier over 8..256 sequences with "
                         "ragged KV lengths in [512, 16384] (one JSON line per point)")
    return ap.parse_args()


# ------------------------------------------------------------------------------------------
# helpers
# ------------------------------------------------------------------------------------------
def max_over_ranks(ms: float, world: int, device) -> float:
    """The job's time: the slowest rank's (every rank runs an independent replica)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank: int, world: int, ms: float) -> float:
    """Whole-job throughput: the tokens of all replicas over the job's time."""
    return world * tokens_per_rank / (ms * 1e-3)


def workload(args):
    """A named workload: synth.WORKLOADS, 'skew' (Zipf routing, block slot map) or
    'sweep_b<N>' (N sequences, ragged KV lengths in [512, 16384])."""
    from intra_spatial_pipelining_gb300 import synth
    if args.workload == "skew":
        wl = synth.skew_workload()
    elif args.workload.startswith("sweep_b"):
        wl = synth.sweep_workload(int(args.workload[len("sweep_b"):]))
    else:
        wl = synth.WORKLOADS[args.workload]
    kw = {}
    if args.layers:
        kw["n_layers"] = args.layers
    if args.kv_len:
        kw["kv_len"] = args.kv_len
    return wl.with_(**kw) if kw else wl


def describe(wl, extra):
    s = wl.shape
    cfg = {"workload": (f"{wl.name}: {wl.n_layers} layers "
                        f"({'alternating sliding-' + str(wl.window) + '/full' if wl.layer_pattern == 'alternate' else 'full'}"
                        f" attention), {wl.n_tokens} sequences, KV {wl.kv_len}, hidden {s.hidden}, "
                        f"{s.n_q_heads}q/{s.n_kv_heads}kv heads x {s.head_dim}, {s.n_experts} experts "
                        f"top-{s.top_k}, {s.n_local_experts} local experts, SwiGLU {s.inter}"
                        + (f", RoPE base {s.rope_theta:g}" if s.rope_theta else "")),
           "layers": wl.n_layers, "n_tokens": wl.n_tokens, "kv_len": wl.kv_len,
           "l2": "inputs larger than L2 (no flush)"}
    cfg.update(extra)
    return cfg


def algorithmic_bytes(wl, kv_lens=None):
    """Unique bytes of one iteration: every weight and KV element read once, the KV append,
    and the per-layer activations (x in/out, a, q, o, h, u, routed rows).  kv_lens: the
    sequences' KV lengths (ragged workloads); default: every sequence at wl.kv_len."""
    s = wl.shape
    per_layer_w = 2 * (s.qkv_rows * s.hidden + s.hidden * s.q_width + s.n_experts * s.hidden
                       + s.n_local_experts * 3 * s.hidden * s.inter + 2 * s.hidden)
    T = wl.n_tokens
    lens = [wl.kv_len] * T if kv_lens is None else [int(v) for v in kv_lens]
    act = 2 * T * (6 * s.hidden + 2 * s.q_width) + T * s.top_k * (2 * s.hidden + 2 * s.inter + 4 * s.hidden)
    tot = 0
    for l in range(wl.n_layers):
        w = wl.layer_window(l)
        positions = sum(min(w, L) if w else L for L in lens)
        kv = s.n_kv_heads * positions * s.head_dim * 2 * 2
        tot += per_layer_w + kv + T * s.n_kv_heads * s.head_dim * 2 * 2 + act
    return tot


def attn_bytes(wl, layer):
    s = wl.shape
    w = wl.layer_window(layer)
    span = min(w, wl.kv_len) if w else wl.kv_len
    T = wl.n_tokens
    return T * s.n_kv_heads * span * s.head_dim * 4 + T * s.q_width * 4


def read_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def read_traffic():
    """ncu DRAM bytes per launch of the attention kernel from the committed summary, or None
    when the summary is missing or was taken from a different kernel source."""
    try:
        txt = open(TRAFFIC_SUMMARY).read()
    except OSError:
        return None
    src_hash = attn_source_hash()
    h = t = None
    for line in txt.splitlines():
        if line.startswith("kernel_source_sha256_16:"):
            h = line.split(":", 1)[1].strip()
        if line.startswith("dram_bytes_per_full_layer_launch:"):
            t = float(line.split(":", 1)[1].strip())
    return t if (h == src_hash and t) else None


def attn_source_hash() -> str:
    """sha256 (first 16 hex digits) of the attention kernel's source files, concatenated."""
    h = hashlib.sha256()
    for f in ATTN_SRCS:
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def blas_threads():
    """Threads of the BLAS thread pool numpy uses (OpenBLAS reports it), or None."""
    import ctypes
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(n[0])
    except Exception:
        pass
    try:
        paths = {ln.split()[-1] for ln in open("/proc/self/maps") if "openblas" in ln.lower()}
    except OSError:
        return None
    for path in sorted(paths):
        try:
            h = ctypes.CDLL(path)
        except OSError:
            continue
        for sym in ("openblas_get_num_threads", "openblas_get_num_threads64_",
                    "scipy_openblas_get_num_threads64_", "scipy_openblas_get_num_threads"):
            f = getattr(h, sym, None)
            if f is not None:
                f.restype = ctypes.c_int
                return int(f())
    return None


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []            # (host arrival time, line)
        self.window = None         # host times bracketing the timed region

    def mark(self, t_begin, t_end):
        self.window = (t_begin, t_end)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lines = self.lines
        if self.window is not None:
            # samples taken while the timed region ran (a line arrives up to one period late)
            t0, t1 = self.window
            inside = [l for t, l in lines if t0 <= t <= t1 + 0.06]
            lines = inside if inside else [l for t, l in lines if t >= t0][:1]
        else:
            lines = [l for _, l in lines]
        for line in lines:
            p = [x.strip() for x in line.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                smax = float(p[2])
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------------------
# CPU oracle (bounded sample)
# ------------------------------------------------------------------------------------------
class OracleSample:
    """The fp64 oracle on a bounded sample: n_tok sequences through one sliding and one full
    layer.  Inputs are drawn once; run() times only the oracle and scales to the metric:
    tokens/s = 1 / (time per token through all layers)."""

    def __init__(self, wl, seed, n_tok=8, layer_pair=(0, 1)):
        import numpy as np

        from intra_spatial_pipelining_gb300 import synth
        from oracle import layer as O
        self.O, self.wl, self.n_tok, self.layer_pair = O, wl, n_tok, layer_pair
        self.x = O.f64(synth.x_in(wl, seed))[:n_tok]
        self.kvl = synth.kv_len(wl, seed).numpy()[:n_tok]
        self.layers = []
        for l in layer_pair:
            w = synth.layer_weights(wl, l, seed)
            caches = [synth.kv_cache_rows(wl, l, seed, b) for b in range(n_tok)]
            kc = np.stack([O.f64(k) for k, _ in caches])
            vc = np.stack([O.f64(v) for _, v in caches])
            self.layers.append((l, w, kc, vc))
        import numpy as np
        np.ones(64) @ np.ones(64)              # load the BLAS before asking for its threads
        self.threads = blas_threads() or os.cpu_count()

    def run(self):
        x = self.x
        t0 = time.perf_counter()
        for l, w, kc, vc in self.layers:
            r = self.O.layer(self.wl.shape, w, x, self.kvl, kc.copy(), vc.copy(),
                             self.wl.layer_window(l))
            x = r["x_next"]
        secs = time.perf_counter() - t0
        per_token_all = secs / self.n_tok * self.wl.n_layers / len(self.layer_pair)
        return 1.0 / per_token_all, secs

    def run_for(self, min_secs):
        """Repeats run() until at least min_secs of oracle time; returns (tokens/s, secs, n)."""
        vals, secs = [], 0.0
        while secs < min_secs or not vals:
            v, t = self.run()
            vals.append(v)
            secs += t
        return statistics.mean(vals), secs, len(vals)

    def describe(self, secs, reps=1):
        return (f"{self.n_tok} sequences through 1 sliding + 1 full layer, {reps} run(s), "
                f"{secs:.1f} s of oracle time (fp64 numpy; a single-threaded per-token loop "
                f"around BLAS calls, BLAS pool of {self.threads} threads), scaled to "
                f"{self.wl.n_layers} layers")


def run_reference(args, rank, world):
    if rank != 0:
        return
    wl = workload(args)
    smp = OracleSample(wl, args.seed, n_tok=4)
    for _ in range(args.warmup):
        smp.run()
    vals, secs = [], 0.0
    for _ in range(args.steps):
        v, t = smp.run()
        vals.append(v)
        secs += t
    value = statistics.mean(vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": describe(wl, {"arm": "fp64 CPU oracle"}),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": smp.threads, "kind": "oracle",
                             "sample": smp.describe(secs, args.steps)},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------------
# secondary shapes: one workload timed pipelined and temporally, then freed
# ------------------------------------------------------------------------------------------
def shape_point(wl, dev, seed, steps, warmup, split=None, micro=None, peak=None,
                cuts=("macro",)):
    """Times one workload on this GPU: the two-stage pipeline (for each cut in `cuts`,
    `split` or the contention-aware balancer's pick checked by full runs of its five best
    candidates; the fastest cut is kept) and temporal execution.  Sliding-window layers share
    one KV buffer: each reads only the last 128 positions of every sequence, so sharing
    changes no timing and halves the memory of the large shapes.  Returns a dict; every
    tensor is freed before it returns."""
    import torch

    from intra_spatial_pipelining_gb300 import sgp, synth
    T = wl.n_tokens
    micro = micro or T // 2
    x = synth.x_in(wl, seed, dev)
    kv_len = synth.kv_len(wl, seed, dev)
    weights = [synth.layer_weights(wl, l, seed, dev) for l in range(wl.n_layers)]
    caches, slide = [], None
    for l in range(wl.n_layers):
        if wl.layer_window(l):
            slide = slide or synth.kv_cache(wl, l, seed, dev)
            caches.append(slide)
        else:
            caches.append(synth.kv_cache(wl, l, seed, dev))
    layers = sgp.layer_array([sgp.make_layer(w, k, v, wl.layer_window(l))
                              for l, (w, (k, v)) in enumerate(zip(weights, caches))])
    d = sgp.make_dims(wl.shape)
    out = x.clone()
    N = sgp.sgp_device_info_get().sm_count
    stream = torch.cuda.current_stream()
    def cut_of(name):
        full = [1] * sgp.N_OPS
        full[sgp.OPS.index("attention")] = 0
        if name == "macro_qkv":
            full[sgp.OPS.index("rmsnorm_attn")] = full[sgp.OPS.index("qkv")] = 0
        return [full, [1] * sgp.N_OPS]

    cut = cut_of(cuts[0])

    def popts(**kw):
        return sgp.make_opts(stage_of_op=cut, stage_lanes=2, **kw)

    def run_ms(nst, spl, mb, opts, n, w):
        p = sgp.sgp_pipeline_create(d, spl, nst, mb, T, wl.cap, opts)
        try:
            for _ in range(w):
                sgp.sgp_pipeline_run(p, layers, kv_len, x, out, T)
            sgp.check(sgp.sgp_pipeline_sync(p), "warm-up")
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(n):
                sgp.sgp_pipeline_run(p, layers, kv_len, x, out, T)
            e1.record(stream)
            e1.synchronize()
            sgp.check(sgp.sgp_pipeline_sync(p), "timed runs")
        finally:
            sgp.sgp_pipeline_destroy(p)
        return e0.elapsed_time(e1) / n

    picked = "given"
    given = split
    best_ms = None
    for name in cuts:
        cut = cut_of(name)
        spl = given
        if spl is None:
            _, rows = sgp.sgp_pipeline_balance(d, layers, kv_len, x, out, T, micro, wl.cap,
                                               quantum=8, reps=2,
                                               opts=popts(stage_times_shared=1))
            cands = [r[0] for r in sorted(rows, key=lambda r: max(r[1], r[2]))[:5]]
            best = min(cands, key=lambda pa: run_ms(2, [pa, N - pa], micro, popts(), 2, 1))
            spl = [best, N - best]
            picked = "contention-aware balancer, best of its 5 best candidates by full runs"
        ms = run_ms(2, spl, micro, popts(), steps, warmup)
        if best_ms is None or ms < best_ms:
            best_ms, split, best_cut = ms, spl, name
    ms_pipe = best_ms
    ms_temp = run_ms(1, [N], T, None, steps, warmup)
    nbytes = algorithmic_bytes(wl, kv_len.cpu().tolist())
    res = {"workload": describe(wl, {})["workload"], "n_tokens": T,
           "sm_split": split, "split_from": picked, "cut": best_cut,
           "microbatch": micro, "lanes_per_stage": 2,
           "pipeline_us": ms_pipe * 1e3, "temporal_us": ms_temp * 1e3,
           "pipeline_speedup": ms_temp / ms_pipe,
           "tokens_per_s_per_gpu": {"pipeline": T / (ms_pipe * 1e-3), "temporal": T / (ms_temp * 1e-3)},
           "tokens_per_s_per_user": {"pipeline": 1e3 / ms_pipe, "temporal": 1e3 / ms_temp},
           "algorithmic_bytes_per_step": nbytes,
           "sliding_layers": "share one KV buffer (timing only)"}
    if peak:
        res["dram_pct_of_peak"] = {"pipeline": 100.0 * nbytes / (ms_pipe * 1e-3) / 1e9 / peak,
                                   "temporal": 100.0 * nbytes / (ms_temp * 1e-3) / 1e9 / peak}
    del layers, x, kv_len, weights, caches, slide, out
    torch.cuda.empty_cache()
    return res


def run_frontier(args):
    """Batch/length sweep: sequences in {8, ..., 256}, ragged KV lengths uniform in
    [512, 16384], 36 alternating layers; one JSON line per point, pipeline (balanced) and
    temporal, tokens/s/user = 1 / iteration and tokens/s/GPU = sequences / iteration."""
    import torch

    from intra_spatial_pipelining_gb300 import sgp, synth
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    sgp.lib()
    synth._CHUNK = 1 << 28
    peak, _ = read_peaks()
    for b in (8, 16, 32, 64, 128, 256):
        wl = synth.sweep_workload(b)
        r = shape_point(wl, dev, args.seed, args.steps, args.warmup, peak=peak,
                        cuts=("macro", "macro_qkv"))
        print(json.dumps({"frontier_point": r}), flush=True)


# ------------------------------------------------------------------------------------------
# GPU arm
# ------------------------------------------------------------------------------------------
def run_sgp(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from intra_spatial_pipelining_gb300 import sgp, synth

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    sgp.lib()
    wl = workload(args)
    s = wl.shape
    T = wl.n_tokens
    seed = args.seed + 1000 * rank

    # ---- inputs (resident in HBM) ----
    synth._CHUNK = 1 << 28
    x = synth.x_in(wl, seed, dev)
    kv_len = synth.kv_len(wl, seed, dev)
    kv_lens = kv_len.cpu().tolist()
    weights = [synth.layer_weights(wl, l, seed, dev) for l in range(wl.n_layers)]
    caches = [synth.kv_cache(wl, l, seed, dev) for l in range(wl.n_layers)]
    layers = sgp.layer_array([sgp.make_layer(w, k, v, wl.layer_window(l))
                              for l, (w, (k, v)) in enumerate(zip(weights, caches))])
    comm = (3.0, 900.0) if args.virtual_comm else (0.0, 0.0)
    d = sgp.make_dims(s, comm_floor_us=comm[0], comm_gbps=comm[1])
    out = x.clone()
    info = sgp.sgp_device_info_get()
    N = info.sm_count
    stream = torch.cuda.current_stream()

    # clock samples are kept only for the timed region; nvidia-smi needs a moment to start
    clocks = ClockSampler(local_rank)
    clocks.start()

    # ---- pipeline configuration ----
    n_stages = args.stages
    micro = args.micro or (T // max(1, wl.microbatches))
    base_kw = {"weight_reuse": 1} if args.weight_reuse else {}
    if n_stages > 1 and args.lanes == 2:
        base_kw["stage_lanes"] = 2

    def cut_kw(cut):
        """Options of a cut (3 stages keep their fixed cut A | B1-B4 | B5-B8)."""
        kw = dict(base_kw)
        if cut in ("macro", "macro_qkv", "macro_oproj") and n_stages == 2:
            full = [1] * sgp.N_OPS
            full[sgp.OPS.index("attention")] = 0
            if cut in ("macro_qkv", "macro_oproj"):
                full[sgp.OPS.index("rmsnorm_attn")] = full[sgp.OPS.index("qkv")] = 0
            if cut == "macro_oproj":
                full[sgp.OPS.index("oproj")] = 0
            kw["stage_of_op"] = [full, [1] * sgp.N_OPS]
        return kw

    def run_ms_opts(spl, o, reps=3):
        p = sgp.sgp_pipeline_create(d, list(spl), len(spl), micro, T, wl.cap, o)
        try:
            sgp.sgp_pipeline_run(p, layers, kv_len, x, out, T)
            sgp.check(sgp.sgp_pipeline_sync(p), "pipeline")
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            t0.record(stream)
            for _ in range(reps):
                sgp.sgp_pipeline_run(p, layers, kv_len, x, out, T)
            t1.record(stream)
            t1.synchronize()
            sgp.check(sgp.sgp_pipeline_sync(p), "pipeline")
        finally:
            sgp.sgp_pipeline_destroy(p)
        return t0.elapsed_time(t1) / reps

    def search_two_stage(cut, sweep):
        """The SM split of a 2-stage cut: the t_A / t_B balancer with stages timed alone and
        under contention, and the Eq. 4-5 makespan from contended task times; each model's best
        candidates (or, with sweep, every legal split) are checked by full pipelined runs."""
        kw = cut_kw(cut)
        o = sgp.make_opts(**kw) if kw else None
        res = {"cut": cut, "full_runs": {}}
        best_alone, rows = sgp.sgp_pipeline_balance(d, layers, kv_len, x, out, T, micro,
                                                    wl.cap, quantum=8, reps=3, opts=o)
        best_shared, rows_shared = sgp.sgp_pipeline_balance(
            d, layers, kv_len, x, out, T, micro, wl.cap, quantum=8, reps=3,
            opts=sgp.make_opts(stage_times_shared=1, **kw))
        # the pages' model (one FIFO per stage): the prediction, checked at its pick by a run
        fifo_opts = sgp.make_opts(**{k: v for k, v in kw.items() if k != "stage_lanes"})
        pred = []
        for r in rows:
            pp = sgp.sgp_pipeline_create(d, [r[0], N - r[0]], 2, micro, T, wl.cap, fifo_opts)
            try:
                t_pred, _ = sgp.sgp_pipeline_predict(pp, layers, kv_len, x, out, T, 2,
                                                     handoff_us=10.0)
            finally:
                sgp.sgp_pipeline_destroy(pp)
            pred.append((r[0], t_pred))
        best_pred = min(pred, key=lambda r: r[1])[0]
        fifo_us = run_ms_opts([best_pred, N - best_pred], fifo_opts) * 1e3

        def full(pa):
            if pa not in res["full_runs"]:
                res["full_runs"][pa] = run_ms_opts([pa, N - pa], o)
            return res["full_runs"][pa]
        if sweep:
            cands = [r[0] for r in rows]
        else:
            cands = [r[0] for r in sorted(pred, key=lambda r: r[1])[:3]]
            for rr in (rows_shared, rows):
                for r in sorted(rr, key=lambda r: max(r[1], r[2]))[:3]:
                    if r[0] not in cands:
                        cands.append(r[0])
        best = min(cands, key=full)
        res.update(split=[best, N - best], ms=full(best), opts_kw=kw, balance=rows,
                   balance_shared=rows_shared, predicted=pred,
                   picks={"alone": best_alone, "shared": best_shared, "predicted": best_pred},
                   fifo_check={"p_A": best_pred, "predicted_us": dict(pred)[best_pred],
                               "measured_us_one_fifo": fifo_us})
        return res

    refine = None
    search = None
    cut_results = None
    opts_kw = cut_kw(args.cut)
    if n_stages == 1:
        split = [N]
    elif args.split in ("auto", "sweep") and n_stages == 2:
        cuts = ["macro", "macro_qkv"] if args.cut == "auto" else [args.cut]
        cut_results = [search_two_stage(c, args.split == "sweep") for c in cuts]
        search = min(cut_results, key=lambda r: r["ms"])
        split, opts_kw = search["split"], search["opts_kw"]
    elif args.split == "auto":
        # 3 stages: pairwise-line refinement (Algorithm 2) on measured full runs, from a uniform
        # seed and from a service-proportional one (SMs in proportion to each stage's work)
        opts = sgp.make_opts(**opts_kw) if opts_kw else None
        a = max(1, info.sm_alignment)
        pmin = max(a, info.sm_min_partition)
        p0 = max(a, (N // 3 // a) * a)
        uni = [p0, p0, N - 2 * p0]
        pp = sgp.sgp_pipeline_create(d, uni, 3, micro, T, wl.cap, opts)
        try:
            t_uni = sgp.sgp_pipeline_stage_times(pp, layers, kv_len, x, out, T, 3, reps=3)
        finally:
            sgp.sgp_pipeline_destroy(pp)
        work = [t * p for t, p in zip(t_uni, uni)]
        prop = [max(pmin, int(round(N * w / sum(work) / a)) * a) for w in work]
        prop[-1] = N - sum(prop[:-1])
        seeds = [uni] + ([prop] if prop != uni and min(prop) >= pmin else [])
        refine = {"seeds": [], "stage_times_uniform_us": t_uni}
        best_t = None
        for sd in seeds:
            spl, t_us, n_ev = sgp.sgp_pipeline_refine(d, layers, kv_len, x, out, T, sd, micro,
                                                      wl.cap, quantum=a, reps=3, opts=opts)
            refine["seeds"].append({"seed": sd, "refined": spl, "us": t_us, "evaluations": n_ev})
            if best_t is None or t_us < best_t:
                best_t, split = t_us, spl
    else:
        split = [int(v) for v in args.split.split(",")]
        if args.cut == "auto":
            opts_kw = cut_kw("macro")
    opts = sgp.make_opts(**opts_kw) if opts_kw else None

    def make(nst, spl, mb, o):
        return sgp.sgp_pipeline_create(d, spl, nst, mb, T, wl.cap, o)

    def time_runs(p, steps, warmup, sampler=None):
        for _ in range(warmup):
            sgp.sgp_pipeline_run(p, layers, kv_len, x, out, T)
        sgp.check(sgp.sgp_pipeline_sync(p), "warmup")
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        t_begin = time.monotonic()
        e0.record(stream)
        for _ in range(steps):
            sgp.sgp_pipeline_run(p, layers, kv_len, x, out, T)
        e1.record(stream)
        torch.cuda.synchronize()
        if sampler is not None:
            sampler.mark(t_begin, time.monotonic())
        sgp.check(sgp.sgp_pipeline_sync(p), "timed runs")
        ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
        if world > 1:
            dist.barrier()
        return ms / steps

    pipe = make(n_stages, split, micro, opts)
    ms_pipe = time_runs(pipe, args.steps, args.warmup, clocks)
    clk = clocks.stop()

    ms_temp = None
    temporal = None
    if not args.no_temporal:
        tp = make(1, [N], T, None)
        ms_temp = time_runs(tp, args.steps, args.warmup)
        sgp.sgp_pipeline_destroy(tp)

    # ---- e2e through the public API: pinned H2D of the step's input, D2H of its result ----
    e2e = None
    if not args.no_e2e:
        hx = x.cpu().pin_memory()
        hout = torch.empty_like(hx).pin_memory()
        x_dev = torch.empty_like(x)
        for _ in range(args.warmup):
            x_dev.copy_(hx, non_blocking=True)
            sgp.sgp_pipeline_run(pipe, layers, kv_len, x_dev, out, T)
            hout.copy_(out, non_blocking=True)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            x_dev.copy_(hx, non_blocking=True)
            sgp.sgp_pipeline_run(pipe, layers, kv_len, x_dev, out, T)
            hout.copy_(out, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        sgp.check(sgp.sgp_pipeline_sync(pipe), "e2e runs")
        ms_e2e = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)
        e2e = {"value": job_tokens_per_s(T, world, ms_e2e), "unit": UNIT,
               "h2d_bytes_per_step": hx.numel() * hx.element_size(),
               "d2h_bytes_per_step": hout.numel() * hout.element_size(),
               "ms_per_step": ms_e2e}
    n_launch, gaps = launches_per_run(make, n_stages, split, micro, opts_kw, layers, kv_len, x,
                                      out, T)
    if args.virtual_comm:  # the communication kernels record no trace: three per layer and microbatch
        n_launch += 3 * wl.n_layers * (T // micro)
    sgp.sgp_pipeline_destroy(pipe)

    # ---- roofline of the dominant kernel (full-attention decode), timed alone ----
    full_layer = next((l for l in range(wl.n_layers) if wl.layer_window(l) == 0), 0)
    lay = layers[full_layer]
    nbytes = sgp.sgp_workspace_bytes(d, T, wl.cap)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
    sgp.sgp_layer_temporal(d, lay, kv_len, x, out, T, None, None, ws, None, stream)
    reps = max(5, args.steps)
    for _ in range(3):
        sgp.sgp_layer_op(d, lay, sgp.OPS.index("attention"), kv_len, x, out, T, ws, stream)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        sgp.sgp_layer_op(d, lay, sgp.OPS.index("attention"), kv_len, x, out, T, ws, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    sgp.check(sgp.sgp_status_from_workspace(ws), "attention launches")
    attn_ms = e0.elapsed_time(e1) / reps
    peak, peak_kind = read_peaks()
    ab = attn_bytes(wl, full_layer)
    achieved = ab / (attn_ms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": read_traffic(),
                "kernel": "attn_decode_kernel (full-attention layer)",
                "algorithmic_bytes_per_launch": ab, "launch_us": attn_ms * 1e3,
                "peak_kind": f"{peak_kind} (MEASURED_PEAKS hbm_gbs copy bandwidth)"}

    paper = None
    if world == 1 and not args.no_paper_shape and args.workload == "gptoss_36l":
        # the pages' own per-GPU decode shape, after the main workload's tensors are freed
        del layers, weights, caches, x, out, ws
        torch.cuda.empty_cache()
        pwl = synth.WORKLOADS["paper_32k"]
        paper = shape_point(pwl, dev, args.seed, max(3, args.steps // 2), 3, split=[56, 96],
                            micro=pwl.n_tokens // 2, peak=read_peaks()[0])
        paper["split_from"] = "fixed 56 | 96 (the balancer's pick at this shape)"
    if rank != 0:
        return
    total_bytes = algorithmic_bytes(wl, kv_lens)
    value = job_tokens_per_s(T, world, ms_pipe)
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        smp = OracleSample(wl, args.seed)
        v, secs, n = smp.run_for(10.0)
        cpu = {"value": v, "unit": UNIT, "cores": smp.threads, "kind": "oracle",
               "sample": smp.describe(secs, n)}
    iter_us = ms_pipe * 1e3
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_pipe, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": describe(wl, {"mode": f"spatial pipeline, {n_stages} stages",
                                "cut": ((search["cut"] if search else args.cut)
                                        if n_stages == 2 else "A | B1-B4 | B5-B8"),
                                "sm_split": split,
                                "microbatches": T // micro, "microbatch": micro,
                                "virtual_comm": ("3 us + payload / 900 GB/s per collective"
                                                 if args.virtual_comm else None),
                                "weight_reuse": bool(args.weight_reuse),
                                "lanes_per_stage": args.lanes if n_stages > 1 else 1,
                                "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}),
        "iteration_us": iter_us,
        "tokens_per_s_per_user": 1e6 / iter_us,
        "dram_algorithmic_gbs": total_bytes / (ms_pipe * 1e-3) / 1e9,
        "dram_pct_of_peak": 100.0 * total_bytes / (ms_pipe * 1e-3) / 1e9 / peak,
        "temporal": None if ms_temp is None else {
            "iteration_us": ms_temp * 1e3, "tokens_per_s": job_tokens_per_s(T, world, ms_temp),
            "dram_pct_of_peak": 100.0 * total_bytes / (ms_temp * 1e-3) / 1e9 / peak,
            "pipeline_speedup": ms_temp / ms_pipe},
        "balance": None if search is None else [
            {"p_A": r[0], "t_A_us": r[1], "t_B_us": r[2]} for r in search["balance"]],
        "balance_shared": None if search is None else [
            {"p_A": r[0], "t_A_us": r[1], "t_B_us": r[2]} for r in search["balance_shared"]],
        "predicted_makespan": None if search is None else {
            "model": "Eq. 4-5 over task durations measured with every stage replaying at once, "
                     "one FIFO per stage, 10 us per cross-stage handoff",
            "rows": [{"p_A": pa, "us": t} for pa, t in search["predicted"]],
            "at_pick": search["fifo_check"]},
        "balancer_picks": None if search is None or args.split == "sweep" else dict(
            search["picks"], chosen=split[0],
            full_run_us={str(k): v * 1e3 for k, v in sorted(search["full_runs"].items())}),
        "cut_search": None if cut_results is None else [
            {"cut": r["cut"], "sm_split": r["split"], "us": r["ms"] * 1e3} for r in cut_results],
        "refine_3_stage": refine,
        "split_sweep": None if search is None or args.split != "sweep" else {
            "balancer_pick": search["picks"]["alone"],
            "sweep_best": split[0],
            "full_run_us": [{"p_A": pa, "us": ms * 1e3}
                            for pa, ms in sorted(search["full_runs"].items())]},
        "roofline": roofline,
        "paper_shape": paper,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps * n_launch,
        "handoff_gap_us": None if gaps is None or len(gaps) == 0 else {
            "median": float(statistics.median(gaps)), "p95": float(sorted(gaps)[int(0.95 * (len(gaps) - 1))]),
            "max": float(max(gaps)), "edges": len(gaps),
            "what": "cross-stage task start minus its data producer's end (graph edge between "
                    "green contexts), from the device launch trace of one run"},
        "clocks": clk,
        "algorithmic_bytes_per_step": total_bytes,
    }
    print(json.dumps(line), flush=True)


def launches_per_run(make, n_stages, split, micro, opts_kw, layers, kv_len, x, out, T):
    """Kernels one pipelined run launches, counted from the device launch trace of a run of
    the same configuration (every kernel records its start; fused ops record nothing), and
    the cross-stage handoff gaps of that run (us)."""
    from intra_spatial_pipelining_gb300 import sgp
    p = make(n_stages, split, micro, sgp.make_opts(trace=1, **opts_kw))
    try:
        sgp.sgp_pipeline_run(p, layers, kv_len, x, out, T)
        sgp.check(sgp.sgp_pipeline_sync(p), "traced run")
        sgp.sgp_pipeline_run(p, layers, kv_len, x, out, T)     # a warm replay
        sgp.check(sgp.sgp_pipeline_sync(p), "traced run")
        tr = sgp.sgp_pipeline_trace(p)
        gaps = sgp.handoff_gaps_us(p).tolist() if n_stages > 1 else None
    finally:
        sgp.sgp_pipeline_destroy(p)
    return int((tr[:, 1] > 0).sum()), gaps


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.frontier:
        run_frontier(args)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        run_sgp(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
