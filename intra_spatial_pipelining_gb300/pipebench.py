"""One run of the layer stack -- pipelined or temporal -- inside a profiler range.

Sets up a workload's stack (its own weights and KV caches), warms the run up, then replays it
once between cudaProfilerStart and cudaProfilerStop, so that a profiler in range mode
measures exactly one iteration, e.g. the DRAM bytes of a whole pipelined iteration against
its algorithmic bytes (the weights that every microbatch reads again show up there):

    python -m intra_spatial_pipelining_gb300.pipebench --layers 2 --split 56,96
    python -m intra_spatial_pipelining_gb300.pipebench --layers 2 --temporal

Prints one JSON line: the mode, the split, the iteration time of the profiled run (CUDA
events) and the algorithmic bytes of one iteration (every weight and KV element once).
"""
from __future__ import annotations

import argparse
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def algorithmic_bytes(wl, kv_lens) -> int:
    """Unique bytes of one iteration, counted as the benchmark counts them: every weight and
    every sequence's KV span read once, the KV append, and the per-layer activations (x in and
    out, a, q, o, h, u; the routed rows, their SwiGLU rows and fp32 expert outputs)."""
    s = wl.shape
    H, T = s.hidden, wl.n_tokens
    w_layer = 2 * (s.qkv_rows * H + H * s.q_width + s.n_experts * H +
                   s.n_local_experts * 3 * H * s.inter + 2 * H)
    per_pos = s.n_kv_heads * s.head_dim * 2 * 2          # K and V, bf16
    act = 2 * T * (6 * H + 2 * s.q_width) + T * s.top_k * (2 * H + 2 * s.inter + 4 * H)
    total = 0
    for l in range(wl.n_layers):
        win = wl.layer_window(l)
        kv = sum(min(L, win) if win else L for L in kv_lens) * per_pos
        total += w_layer + kv + T * per_pos + act
    return total


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="gptoss_36l")
    ap.add_argument("--layers", type=int, default=2)
    ap.add_argument("--temporal", action="store_true", help="one stage on every SM")
    ap.add_argument("--split", default="56,96", help="SMs of stage A, stage B")
    ap.add_argument("--cut", default="macro_qkv", choices=["macro", "macro_qkv", "layer"])
    ap.add_argument("--micro", type=int, default=None, help="sequences per microbatch")
    ap.add_argument("--weight-reuse", action="store_true",
                    help="L2 evict-last hint on the weights a later microbatch reads again")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--seed", type=int, default=0)
    args = ap.parse_args()

    import torch

    from intra_spatial_pipelining_gb300 import sgp, synth
    wl = synth.WORKLOADS[args.workload].with_(n_layers=args.layers)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    sgp.lib()
    T = wl.n_tokens
    x = synth.x_in(wl, args.seed, dev)
    kv_len = synth.kv_len(wl, args.seed, dev)
    weights = [synth.layer_weights(wl, l, args.seed, dev) for l in range(wl.n_layers)]
    caches = [synth.kv_cache(wl, l, args.seed, dev) for l in range(wl.n_layers)]
    layers = sgp.layer_array([sgp.make_layer(w, k, v, wl.layer_window(l))
                              for l, (w, (k, v)) in enumerate(zip(weights, caches))])
    d = sgp.make_dims(wl.shape)
    out = torch.empty_like(x)
    N = sgp.sgp_device_info_get().sm_count
    if args.temporal:
        split, micro, opts = [N], T, None
    else:
        split = [int(v) for v in args.split.split(",")]
        micro = args.micro or T // 2
        full = [1] * sgp.N_OPS
        if args.cut == "layer":
            full[0] = full[1] = full[2] = 0
            slide = list(full)
        else:
            full[sgp.OPS.index("attention")] = 0
            if args.cut == "macro_qkv":
                full[sgp.OPS.index("rmsnorm_attn")] = full[sgp.OPS.index("qkv")] = 0
            slide = [1] * sgp.N_OPS
        opts = sgp.make_opts(stage_of_op=[full, slide], stage_lanes=2,
                             **({"weight_reuse": 1} if args.weight_reuse else {}))
    p = sgp.sgp_pipeline_create(d, split, len(split), micro, T, wl.cap, opts)
    try:
        for _ in range(args.warmup):
            sgp.sgp_pipeline_run(p, layers, kv_len, x, out, T)
        sgp.check(sgp.sgp_pipeline_sync(p), "warm-up")
        stream = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        torch.cuda.profiler.start()
        e0.record(stream)
        sgp.sgp_pipeline_run(p, layers, kv_len, x, out, T)
        e1.record(stream)
        e1.synchronize()
        sgp.check(sgp.sgp_pipeline_sync(p), "profiled run")
        torch.cuda.synchronize()
        torch.cuda.profiler.stop()
    finally:
        sgp.sgp_pipeline_destroy(p)
    print(json.dumps({"mode": "temporal" if args.temporal else "pipeline", "workload": wl.name,
                      "layers": wl.n_layers, "n_tokens": T, "sm_split": split,
                      "microbatch": micro, "cut": None if args.temporal else args.cut,
                      "weight_reuse": bool(args.weight_reuse),
                      "run_us": e0.elapsed_time(e1) * 1e3,
                      "algorithmic_bytes": algorithmic_bytes(wl, kv_len.cpu().tolist())}),
          flush=True)


if __name__ == "__main__":
    main()
