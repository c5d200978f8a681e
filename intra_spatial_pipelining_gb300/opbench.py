"""Per-operator timing of one decode layer through the C ABI (sgp_layer_op).

One layer of a named workload is set up on the GPU (its own weights and KV cache only),
run once temporally so that the workspace holds every intermediate, and then one operator
(``--op``) is launched ``--reps`` times alone.  Each launch recomputes that operator from
the same inputs, so the launches are identical.  The line printed per operator gives its
CUDA-event time, its algorithmic bytes (every weight and KV element once, plus its
activations) and the bandwidth those bytes imply.

Used to time and profile single kernels, e.g. a profiler restricted to one kernel name
skips the launches of the set-up layer and captures the first launch of the operator:

    python -m intra_spatial_pipelining_gb300.opbench --op qkv --reps 3
    python -m intra_spatial_pipelining_gb300.opbench --op all --tokens 8 --path gemv

    ops: rmsnorm_attn qkv attention oproj router dispatch expert_up expert_down combine
"""
from __future__ import annotations

import argparse
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def op_bytes(wl, layer: int, op: str, n_tokens: int) -> int:
    """Algorithmic bytes of one operator of one layer: its weights and KV once, plus the
    activations it reads and writes (bf16 unless stated)."""
    s = wl.shape
    T, H, k = n_tokens, s.hidden, s.top_k
    R = T * k
    win = wl.layer_window(layer)
    span = min(win, wl.kv_len) if win else wl.kv_len
    if op == "rmsnorm_attn":
        return 2 * (2 * T * H + H)
    if op == "qkv":
        return 2 * (s.qkv_rows * H + T * H + T * s.q_width + 2 * T * s.n_kv_heads * s.head_dim)
    if op == "attention":
        return (T * s.n_kv_heads * span * s.head_dim * 2 * 2) + 2 * 2 * T * s.q_width
    if op == "oproj":
        return 2 * (H * s.q_width + T * s.q_width + 2 * T * H)
    if op == "router":
        return 2 * (s.n_experts * H + 2 * T * H + H) + 4 * T * s.n_experts + 8 * R
    if op == "dispatch":
        return 2 * 2 * R * H + 4 * R
    if op == "expert_up":
        return 2 * (s.n_local_experts * 2 * s.inter * H + R * H + R * s.inter)
    if op == "expert_down":
        return 2 * (s.n_local_experts * H * s.inter + R * s.inter) + 4 * R * H
    if op == "combine":
        return 2 * 2 * T * H + 4 * R * H + 8 * R
    raise ValueError(op)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="gptoss_36l")
    ap.add_argument("--layer", type=int, default=1, help="layer index (sets the window)")
    ap.add_argument("--tokens", type=int, default=None, help="override the sequence count")
    ap.add_argument("--op", default="all")
    ap.add_argument("--reps", type=int, default=20)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--path", default="auto", choices=["auto", "gemv", "tc"],
                    help="projection path (auto: the library's default threshold)")
    args = ap.parse_args()

    import torch

    from intra_spatial_pipelining_gb300 import sgp, synth

    wl = synth.WORKLOADS[args.workload]
    if args.tokens:
        wl = wl.with_(n_tokens=args.tokens)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    sgp.lib()
    T = wl.n_tokens
    x = synth.x_in(wl, args.seed, dev)
    kv_len = synth.kv_len(wl, args.seed, dev)
    w = synth.layer_weights(wl, args.layer, args.seed, dev)
    kc, vc = synth.kv_cache(wl, args.layer, args.seed, dev)
    layer = sgp.make_layer(w, kc, vc, wl.layer_window(args.layer))
    d = sgp.make_dims(wl.shape, {"auto": sgp.PATH_AUTO, "gemv": sgp.PATH_GEMV,
                                 "tc": sgp.PATH_TC}[args.path])
    ws = torch.zeros(sgp.sgp_workspace_bytes(d, T, wl.cap), dtype=torch.uint8, device=dev)
    out = torch.empty_like(x)
    stream = torch.cuda.current_stream()
    sgp.sgp_layer_temporal(d, layer, kv_len, x, out, T, None, None, ws, None, stream)
    sgp.check(sgp.sgp_status_from_workspace(ws), "set-up layer")
    ops = sgp.OPS if args.op == "all" else (args.op,)
    for name in ops:
        op = sgp.OPS.index(name)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.reps):
            sgp.sgp_layer_op(d, layer, op, kv_len, x, out, T, ws, stream)
        e1.record(stream)
        e1.synchronize()
        sgp.check(sgp.sgp_status_from_workspace(ws), name)
        us = e0.elapsed_time(e1) * 1e3 / args.reps
        nb = op_bytes(wl, args.layer, name, T)
        print(json.dumps({"op": name, "workload": wl.name, "layer": args.layer,
                          "window": wl.layer_window(args.layer), "n_tokens": T,
                          "us_per_launch": us, "algorithmic_bytes": nb,
                          "algorithmic_gbs": nb / (us * 1e-6) / 1e9}), flush=True)


if __name__ == "__main__":
    main()
