"""fp64 CPU oracle of one MoE decode layer and of an L-layer decode stack.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only the tests, the smoke check in ``__graft_entry__`` and
the CPU-baseline leg of ``bench.py`` use it.  It shares no code with the CUDA
path; its only shared input is the seeded generator, which holds none of the
layer's arithmetic.

What it computes (plain definitions, numpy float64, no blocking or fusion):
the operator chain of one MoE transformer decode layer as listed in
"SubGPU Pipelining: Intra-GPU Fine-Grained Spatial Parallelism for LLM
Inference", Fig. 3 (RMSNorm, Q/KV projection, FMHA, output projection,
Add+Norm, router gating, TopK, dispatch, expert up + SwiGLU, expert down,
combine), with the stage contents of the two-stage cut (stage A: RMSNorm, QKV
projection, attention; stage B: output projection + residual, RMSNorm, router
top-k, SwiGLU experts, weighted combine).  Sliding-window and full-attention
layers alternate as described in Section 5.1 of the same paper.

Where the page leaves a step open, the readings are:
  * RMSNorm: y = x / sqrt(mean(x^2) + eps) * g, eps = 1e-5.
  * No biases, no attention sinks, plain SwiGLU silu(gate) * up.  RoPE only when
    the shape sets rope_theta > 0 (half-split pairs, applied to q and k_new at
    position L-1 before rounding; cached keys are taken as already rotated).
  * The current token's k, v are written to cache slot L-1 (L = kv_len counts
    the current token); attention runs over [lo, L), lo = max(0, L - W) for a
    sliding window W, else 0.  Scale 1/sqrt(d).  Query head h reads KV head
    h // (n_q / n_kv).
  * Router: logits z = u W_r^T (+ bias), top-k by descending logit with ties to
    the lower index, weights = softmax over the k selected logits.
  * Expert-parallel loopback: global expert g is served by local weight slot
    g mod E_local ("mod") or g * E_local // E ("block").
  * Combine: x_next = h + sum_j w_j y_j (pre-norm residual).
  * bf16 rounding (round to nearest even) is applied at exactly the tensors
    the GPU stores in bf16: a, q, k, v (and the cache write), o, h, u, the
    SwiGLU output and x_next.  Router logits, top-k weights and expert-down
    outputs stay unrounded (the GPU keeps them in fp32).
"""
from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------------------
# bf16 rounding
# ---------------------------------------------------------------------------
_DROP = 45                                   # fp64 has 52 fraction bits, bf16 has 7
_HALF = np.uint64((1 << (_DROP - 1)) - 1)
_MASK = np.uint64(~((1 << _DROP) - 1) & 0xFFFFFFFFFFFFFFFF)


def bf16(x) -> np.ndarray:
    """Round float64 values to the nearest bf16 value, ties to even (result is float64)."""
    x = np.asarray(x, dtype=np.float64)
    u = np.ascontiguousarray(x).reshape(-1).view(np.uint64)
    lsb = (u >> np.uint64(_DROP)) & np.uint64(1)
    r = ((u + _HALF + lsb) & _MASK).view(np.float64)
    return r.reshape(x.shape)


def f64(t) -> np.ndarray:
    """A torch tensor (any float dtype, any device) or array as float64 numpy."""
    if hasattr(t, "detach"):
        import torch
        return t.detach().to("cpu", torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


# ---------------------------------------------------------------------------
# operators (each a plain definition)
# ---------------------------------------------------------------------------
def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * g (unrounded)."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * g


def linear(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """y = x W^T for W stored [out][in]."""
    return x @ w.T


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, lo: int, hi: int) -> np.ndarray:
    """One query head over positions [lo, hi): softmax(q K^T / sqrt(d)) V (unrounded).

    q [d], k/v [positions][d]."""
    d = q.shape[-1]
    s = (k[lo:hi] @ q) / np.sqrt(d)
    s = s - np.max(s)
    p = np.exp(s)
    p = p / np.sum(p)
    return p @ v[lo:hi]


def rope(x: np.ndarray, pos: int, theta: float) -> np.ndarray:
    """Rotary position embedding of head vectors x [..][d] at position ``pos`` (unrounded).

    Dimension pairs (i, i + d/2), i < d/2, are rotated by the angle pos * theta^(-2i/d)
    (the half-split pairing; "SubGPU Pipelining: Intra-GPU Fine-Grained Spatial Parallelism
    for LLM Inference", Fig. 3 lists RoPE in the operator chain without its variant)."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    half = d // 2
    freq = theta ** (-2.0 * np.arange(half) / d)
    ang = pos * freq
    c, s_ = np.cos(ang), np.sin(ang)
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s_, a * s_ + b * c], axis=-1)


def topk(z: np.ndarray, k: int):
    """Indices of the k largest logits (descending, ties to the lower index) and
    the softmax over the selected logits."""
    order = sorted(range(z.shape[0]), key=lambda e: (-z[e], e))[:k]
    sel = np.array([z[e] for e in order])
    p = np.exp(sel - np.max(sel))
    return np.array(order, dtype=np.int64), p / np.sum(p)


def topk_margin(z: np.ndarray, k: int) -> float:
    """Gap between the k-th and (k+1)-th largest logit of one token."""
    s = np.sort(z)[::-1]
    return float(s[k - 1] - s[k]) if s.shape[0] > k else float("inf")


def slot_of(g: int, n_experts: int, n_local: int, slot_map: str) -> int:
    if slot_map == "mod":
        return g % n_local
    if slot_map == "block":
        return g * n_local // n_experts
    raise ValueError(slot_map)


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def swiglu_expert(u: np.ndarray, w_gate_up: np.ndarray, w_down: np.ndarray, inter: int):
    """One expert on one token: z = bf16(silu(u Wg^T) * (u Wu^T)), y = z Wd^T.

    w_gate_up is [2*inter][H] (gate rows then up rows), w_down is [H][inter]."""
    gate = w_gate_up[:inter] @ u
    up = w_gate_up[inter:] @ u
    z = bf16(silu(gate) * up)
    return z, w_down @ z


# ---------------------------------------------------------------------------
# the layer
# ---------------------------------------------------------------------------
def layer(shape, weights: dict, x: np.ndarray, kv_len: np.ndarray, k_cache: np.ndarray,
          v_cache: np.ndarray, window: int, tokens=None) -> dict:
    """One decode layer for the tokens listed in ``tokens`` (default: all).

    ``x`` is [T][H] (bf16 values held in float64).  ``k_cache``/``v_cache`` are
    indexed [token][kv_head][pos][d] and are updated IN PLACE at position
    kv_len[t]-1 for the listed tokens.  Returns a dict of per-token results,
    each an array whose first axis follows ``tokens``.
    """
    H, d = shape.hidden, shape.head_dim
    nq, nkv = shape.n_q_heads, shape.n_kv_heads
    grp = nq // nkv
    I, k = shape.inter, shape.top_k
    if tokens is None:
        tokens = list(range(x.shape[0]))
    W = {n: (f64(v) if v is not None else None) for n, v in weights.items()}

    out = {n: [] for n in ("a", "q", "k_new", "v_new", "o", "h", "u", "logits",
                           "idx", "w", "slot", "z", "y", "x_next")}
    for t in tokens:
        xt = x[t]
        # stage A: RMSNorm -> QKV projection -> KV append -> attention
        a = bf16(rmsnorm(xt, W["g_attn"], shape.rms_eps))
        qkv = linear(a, W["w_qkv"])
        L = int(kv_len[t])
        qr = qkv[: nq * d].reshape(nq, d)
        kr = qkv[nq * d:(nq + nkv) * d].reshape(nkv, d)
        theta = getattr(shape, "rope_theta", 0.0)
        if theta:
            # the new token sits at position L-1; cached keys are already rotated
            qr, kr = rope(qr, L - 1, theta), rope(kr, L - 1, theta)
        q = bf16(qr)
        kn = bf16(kr)
        vn = bf16(qkv[(nq + nkv) * d:]).reshape(nkv, d)
        k_cache[t, :, L - 1, :] = kn
        v_cache[t, :, L - 1, :] = vn
        lo = max(0, L - window) if window > 0 else 0
        o = np.empty((nq, d))
        for h in range(nq):
            o[h] = attention(q[h], k_cache[t, h // grp], v_cache[t, h // grp], lo, L)
        o = bf16(o).reshape(nq * d)
        # stage B: output projection + residual -> RMSNorm -> router -> experts -> combine
        hres = bf16(xt + linear(o, W["w_o"]))
        u = bf16(rmsnorm(hres, W["g_mlp"], shape.rms_eps))
        z = linear(u, W["w_router"])
        if W.get("router_bias") is not None:
            z = z + W["router_bias"]
        idx, wt = topk(z, k)
        acc = np.zeros(H)
        zs, ys, slots = [], [], []
        for j in range(k):
            s = slot_of(int(idx[j]), shape.n_experts, shape.n_local_experts, shape.slot_map)
            zz, yy = swiglu_expert(u, W["w_gate_up"][s], W["w_down"][s], I)
            acc = acc + wt[j] * yy
            zs.append(zz)
            ys.append(yy)
            slots.append(s)
        xn = bf16(hres + acc)
        for n, v in (("a", a), ("q", q.reshape(-1)), ("k_new", kn), ("v_new", vn), ("o", o),
                     ("h", hres), ("u", u), ("logits", z), ("idx", idx), ("w", wt),
                     ("slot", np.array(slots)), ("z", np.array(zs)), ("y", np.array(ys)),
                     ("x_next", xn)):
            out[n].append(v)
    return {n: np.array(v) for n, v in out.items()}


def stack(shape, layers_weights: list, windows: list, x: np.ndarray, kv_len: np.ndarray,
          caches: list, tokens=None) -> dict:
    """L layers back to back: layer l's x_next feeds layer l+1.

    ``caches`` is a list of (k_cache, v_cache) per layer, updated in place.
    Returns {"x_out": [T'][H], "idx": [L][T'][k], "w": [L][T'][k], "logits": [L][T'][E]}."""
    if tokens is None:
        tokens = list(range(x.shape[0]))
    cur = np.array(x, dtype=np.float64)
    idxs, ws, zs = [], [], []
    for li, (wts, win) in enumerate(zip(layers_weights, windows)):
        r = layer(shape, wts, cur, kv_len, caches[li][0], caches[li][1], win, tokens)
        nxt = cur.copy()
        nxt[tokens] = r["x_next"]
        cur = nxt
        idxs.append(r["idx"])
        ws.append(r["w"])
        zs.append(r["logits"])
    return {"x_out": cur[tokens], "idx": np.array(idxs), "w": np.array(ws),
            "logits": np.array(zs)}
