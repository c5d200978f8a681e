"""Shared helpers of the GPU parity tests and of ``__graft_entry__.smoke()``.

Inputs come from the seeded generator only; expected values come from the fp64
oracle only.  The CUDA path is reached through the C-ABI binding.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

from intra_spatial_pipelining_gb300 import sgp, synth
from oracle import layer as O

MARGIN = 1e-3        # minimum top-k logit gap kept by the generator's resampling
TOL = 2e-2           # bf16 tensors: max|err| <= TOL * max|ref| per tensor


@dataclasses.dataclass
class Inputs:
    wl: synth.Workload
    seed: int
    x: torch.Tensor            # device bf16 [T][H]
    kv_len: torch.Tensor       # device int32 [T]
    weights: list              # per layer dict of device tensors
    caches: list               # per layer (k, v) device bf16
    attempts: list             # router resampling attempt per layer

    @property
    def shape(self):
        return self.wl.shape

    def sgp_layers(self):
        return [sgp.make_layer(w, k, v, self.wl.layer_window(l))
                for l, (w, (k, v)) in enumerate(zip(self.weights, self.caches))]

    def fresh_caches(self):
        """Device caches re-drawn from the generator (undoes KV appends)."""
        return [synth.kv_cache(self.wl, l, self.seed, "cuda") for l in range(self.wl.n_layers)]

    def reset_caches(self):
        for (k, v), (k0, v0) in zip(self.caches, self.fresh_caches()):
            k.copy_(k0)
            v.copy_(v0)


def make_inputs(wl: synth.Workload, seed: int, attempts=None, device="cuda") -> Inputs:
    attempts = list(attempts) if attempts is not None else [0] * wl.n_layers
    x = synth.x_in(wl, seed, device)
    kvl = synth.kv_len(wl, seed, device)
    ws = [synth.layer_weights(wl, l, seed, device, router_attempt=attempts[l])
          for l in range(wl.n_layers)]
    cs = [synth.kv_cache(wl, l, seed, device) for l in range(wl.n_layers)]
    return Inputs(wl, seed, x, kvl, ws, cs, attempts)


def oracle_stack(inp: Inputs, tokens=None) -> dict:
    """fp64 oracle of the whole stack (per-token results for ``tokens``)."""
    wl = inp.wl
    ws = [{n: (v.cpu() if v is not None else None) for n, v in w.items()} for w in inp.weights]
    caches = []
    for l in range(wl.n_layers):
        k, v = synth.kv_cache(wl, l, inp.seed, "cpu")
        caches.append((O.f64(k), O.f64(v)))
    return O.stack(wl.shape, ws, [wl.layer_window(l) for l in range(wl.n_layers)],
                   O.f64(inp.x), inp.kv_len.cpu().numpy(), caches, tokens)


def oracle_layer(inp: Inputs, layer: int = 0, x=None, tokens=None) -> dict:
    wl = inp.wl
    w = {n: (v.cpu() if v is not None else None) for n, v in inp.weights[layer].items()}
    k, v = synth.kv_cache(wl, layer, inp.seed, "cpu")
    kc, vc = O.f64(k), O.f64(v)
    xx = O.f64(inp.x) if x is None else x
    return O.layer(wl.shape, w, xx, inp.kv_len.cpu().numpy(), kc, vc, wl.layer_window(layer),
                   tokens)


def make_inputs_with_margin(wl: synth.Workload, seed: int, max_attempts: int = 20):
    """Single-layer workloads: redraw the router weights (attempt index) until every
    token's oracle top-k margin is >= MARGIN.  Returns (inputs, oracle result)."""
    assert wl.n_layers == 1
    for a in range(max_attempts):
        inp = make_inputs(wl, seed, [a])
        ref = oracle_layer(inp)
        m = min(O.topk_margin(z, wl.shape.top_k) for z in ref["logits"])
        if m >= MARGIN:
            return inp, ref
    raise RuntimeError("no router draw with the required margin")


def make_stack_inputs_with_margin(wl: synth.Workload, seed: int, tokens=None,
                                  max_attempts: int = 30):
    """Multi-layer workloads: redraw the router weights of the first layer whose oracle
    top-k margin (over ``tokens``) is below MARGIN, until every layer keeps the margin.
    Returns (inputs, oracle result of the stack for ``tokens``)."""
    attempts = [0] * wl.n_layers
    for _ in range(max_attempts):
        inp = make_inputs(wl, seed, attempts)
        ref = oracle_stack(inp, tokens)
        bad = [l for l in range(wl.n_layers)
               if min(O.topk_margin(z, wl.shape.top_k) for z in ref["logits"][l]) < MARGIN]
        if not bad:
            return inp, ref
        attempts[bad[0]] += 1
    raise RuntimeError("no router draws with the required margin")


def oracle_stack_rows(inp: Inputs, seqs) -> dict:
    """fp64 oracle of the whole stack for the sequences ``seqs`` only (every result of a
    sequence depends on that sequence alone).  The layer weights and those sequences' KV rows
    are copied from the generator's tensors one layer at a time, so the full-size stack never
    has to be held on the host."""
    wl = inp.wl
    x = O.f64(inp.x.cpu())[seqs]
    kvl = inp.kv_len.cpu().numpy()[seqs]
    idxs, ws, zs = [], [], []
    for l in range(wl.n_layers):
        w = {n: (v.cpu() if v is not None else None) for n, v in inp.weights[l].items()}
        k, v = inp.caches[l]
        kc, vc = O.f64(k[seqs].cpu()), O.f64(v[seqs].cpu())
        r = O.layer(wl.shape, w, x, kvl, kc, vc, wl.layer_window(l))
        x = r["x_next"]
        idxs.append(r["idx"])
        ws.append(r["w"])
        zs.append(r["logits"])
    return {"x_out": x, "idx": np.array(idxs), "w": np.array(ws), "logits": np.array(zs)}


def rel_err(gpu, ref) -> float:
    g = gpu.detach().to("cpu", torch.float64).numpy() if hasattr(gpu, "detach") else np.asarray(gpu)
    r = np.asarray(ref, dtype=np.float64).reshape(g.shape)
    den = max(np.max(np.abs(r)), 1e-30)
    return float(np.max(np.abs(g - r)) / den)


def assert_close(name, gpu, ref, tol=TOL):
    e = rel_err(gpu, ref)
    assert e <= tol, f"{name}: max|err|/max|ref| = {e:.3e} > {tol}"
    return e


def routing_sets(idx) -> list:
    a = idx.detach().cpu().numpy() if hasattr(idx, "detach") else np.asarray(idx)
    return [tuple(sorted(int(v) for v in row)) for row in a.reshape(-1, a.shape[-1])]


def dims(shape, path=sgp.PATH_AUTO, gemv_max_tokens=16):
    """The tests' threshold (16) keeps their 6-12-sequence cases on the GEMV path, so both
    projection paths are covered; the library's default is lower."""
    return sgp.make_dims(shape, path, gemv_max_tokens)


def workspace(d, n_tokens, max_kv):
    nbytes = sgp.sgp_workspace_bytes(d, n_tokens, max_kv)
    assert nbytes > 0
    return torch.zeros(nbytes, dtype=torch.uint8, device="cuda")


def dump_buffers(shape, T):
    H, qw, k = shape.hidden, shape.q_width, shape.top_k
    R = T * k
    bf = dict(dtype=torch.bfloat16, device="cuda")
    b = {"a": torch.zeros(T, H, **bf), "q": torch.zeros(T, qw, **bf), "o": torch.zeros(T, qw, **bf),
         "h": torch.zeros(T, H, **bf), "u": torch.zeros(T, H, **bf),
         "logits": torch.zeros(T, shape.n_experts, dtype=torch.float32, device="cuda"),
         "slot_offsets": torch.zeros(shape.n_local_experts + 1, dtype=torch.int32, device="cuda"),
         "pair_pos": torch.zeros(R, dtype=torch.int32, device="cuda"),
         "z": torch.zeros(R, shape.inter, **bf),
         "y": torch.zeros(R, H, dtype=torch.float32, device="cuda")}
    st = sgp.sgp_layer_dump(*[b[n].data_ptr() for n in ("a", "q", "o", "h", "u", "logits",
                                                       "slot_offsets", "pair_pos", "z", "y")])
    return b, st


def run_temporal_layer(inp: Inputs, d, layer: int = 0, dump=True):
    wl = inp.wl
    T = wl.n_tokens
    ws = workspace(d, T, wl.cap)
    out = torch.empty_like(inp.x)
    tki = torch.full((T, wl.shape.top_k), -1, dtype=torch.int32, device="cuda")
    tkw = torch.zeros(T, wl.shape.top_k, dtype=torch.float32, device="cuda")
    bufs, st = dump_buffers(wl.shape, T) if dump else (None, None)
    lay = inp.sgp_layers()[layer]
    sgp.sgp_layer_temporal(d, lay, inp.kv_len, inp.x, out, T, tki, tkw, ws, st)
    status = sgp.sgp_status_from_workspace(ws)
    return {"x_next": out, "idx": tki, "w": tkw, "dump": bufs, "status": status, "ws": ws}
