"""Seeded synthetic inputs for the decode layer (weights, KV cache, activations).

This module is shared by the CUDA path (bench, GPU tests) and by the CPU
oracle's tests, so it deliberately holds none of the layer's arithmetic: it only
draws numbers.  Every value is a pure function of (seed, tensor name, layer,
flat element index), computed with integer hashing plus one exactly-rounded
fp32 multiply and a round-to-nearest-even bf16 conversion.  The same call
therefore gives bit-identical tensors on the CPU and on a GPU, and any slice of
a tensor (for example one sequence's KV rows) can be drawn on its own.

Distribution: "normal" values use the Irwin-Hall sum of four 16-bit uniforms
(mean 0, unit variance after scaling, tails cut at about 3.46 sigma).  It
stands in for N(0, sigma) without transcendental functions, whose last-ulp
behaviour differs between CPU and GPU libraries.

The workload shapes follow the per-GPU slice of GPT-OSS-120B decode described
in "SubGPU Pipelining: Intra-GPU Fine-Grained Spatial Parallelism for LLM
Inference", Section 5.1 (TP8/DP4 attention, EP32 MoE, global batch 2,048),
scaled to 64 sequences x 8 KV heads per GPU.
"""
from __future__ import annotations

import dataclasses
import math
import zlib
from typing import Optional

import torch

M32 = 0xFFFFFFFF
# standard deviation of the sum of four independent uniforms on {0..65535}
_IH4_STD = math.sqrt((65536.0 * 65536.0 - 1.0) / 3.0)
_IH4_MEAN = 2 * 65535


# --------------------------------------------------------------------------
# counter-based hashing (torch int64 arithmetic, values kept in [0, 2**32))
# --------------------------------------------------------------------------
def _mul32(x: torch.Tensor, c: int) -> torch.Tensor:
    """(x * c) mod 2**32 for x in [0, 2**32) without int64 overflow."""
    lo = x * (c & 0xFFFF)
    hi = ((x * (c >> 16)) & 0xFFFF) << 16
    return (lo + hi) & M32


def _lowbias32(x: torch.Tensor) -> torch.Tensor:
    """32-bit integer mixer (xorshift-multiply, constants 0x7feb352d / 0x846ca68b)."""
    x = x ^ (x >> 16)
    x = _mul32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32(x, 0x846CA68B)
    x = x ^ (x >> 16)
    return x


def _mix_py(x: int) -> int:
    """Host-side copy of the mixer for deriving per-tensor keys."""
    x &= M32
    x ^= x >> 16
    x = (x * 0x7FEB352D) & M32
    x ^= x >> 15
    x = (x * 0x846CA68B) & M32
    x ^= x >> 16
    return x


def tensor_key(seed: int, name: str, layer: int = 0) -> tuple[int, int]:
    """Two 32-bit keys for one named tensor of one layer."""
    base = _mix_py(zlib.crc32(name.encode()) ^ _mix_py(seed & M32) ^ _mix_py((seed >> 32) + 0x9E37))
    base = _mix_py(base ^ _mix_py(layer * 0x85EBCA6B + 0x27D4EB2F))
    return base, _mix_py(base ^ 0x5BD1E995)


def _hash_pair(idx: torch.Tensor, keys: tuple[int, int]) -> tuple[torch.Tensor, torch.Tensor]:
    ha = _lowbias32((idx + keys[0]) & M32)
    hb = _lowbias32(ha ^ keys[1])
    return ha, hb


def _indices(start: int, count: int, device) -> torch.Tensor:
    if start < 0 or start + count > (1 << 32):
        raise ValueError("tensor too large for the 32-bit element counter")
    return torch.arange(start, start + count, dtype=torch.int64, device=device)


_CHUNK = 1 << 26


def normal_flat(seed: int, name: str, layer: int, start: int, count: int,
                sigma: float, device="cpu", mean_one: bool = False) -> torch.Tensor:
    """bf16 values ~N(0, sigma) (or 1 + N(0, sigma)) for flat indices [start, start+count)."""
    out = torch.empty(count, dtype=torch.bfloat16, device=device)
    keys = tensor_key(seed, name, layer)
    scale = torch.tensor(sigma / _IH4_STD, dtype=torch.float32, device=device)
    one = torch.tensor(1.0, dtype=torch.float32, device=device)
    for off in range(0, count, _CHUNK):
        n = min(_CHUNK, count - off)
        ha, hb = _hash_pair(_indices(start + off, n, device), keys)
        s = (ha & 0xFFFF) + (ha >> 16) + (hb & 0xFFFF) + (hb >> 16) - _IH4_MEAN
        v = s.to(torch.float32) * scale          # exact int -> fp32, one rounded multiply
        if mean_one:
            v = v + one
        out[off:off + n] = v.to(torch.bfloat16)  # round to nearest even
        del ha, hb, s, v
    return out


def normal(seed: int, name: str, layer: int, shape, sigma: float, device="cpu",
           mean_one: bool = False) -> torch.Tensor:
    n = 1
    for s in shape:
        n *= int(s)
    return normal_flat(seed, name, layer, 0, n, sigma, device, mean_one).view(*shape)


def uniform_int(seed: int, name: str, layer: int, count: int, lo: int, hi: int,
                device="cpu") -> torch.Tensor:
    """int32 values uniform on [lo, hi] (inclusive), modulo bias < 2**-16."""
    ha, hb = _hash_pair(_indices(0, count, device), tensor_key(seed, name, layer))
    span = hi - lo + 1
    return (lo + (((ha << 16) ^ (hb & 0xFFFF)) % span)).to(torch.int32)


# --------------------------------------------------------------------------
# workload descriptions
# --------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class LayerShape:
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    n_experts: int
    top_k: int
    n_local_experts: int
    inter: int
    rms_eps: float = 1e-5
    slot_map: str = "mod"          # "mod": g % E_local, "block": g * E_local // E
    rope_theta: float = 0.0        # RoPE base (0: no rotation)

    @property
    def qkv_rows(self) -> int:
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim

    @property
    def q_width(self) -> int:
        return self.n_q_heads * self.head_dim


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    shape: LayerShape
    n_tokens: int                  # sequences in the decode batch (one token each)
    n_layers: int
    kv_len: int                    # uniform KV length (counting the current token)
    kv_len_range: Optional[tuple[int, int]] = None   # ragged lengths when set
    kv_cap: int = 0                # allocated positions per sequence (0 = max length)
    window: int = 128              # sliding-window length for sliding layers
    layer_pattern: str = "full"    # "full" | "alternate" (even sliding, odd full)
    w_sigma: float = 0.02
    x_sigma: float = 1.0
    kv_sigma: float = 0.02
    microbatches: int = 2
    zipf_bias: float = 0.0         # router bias -s*ln(g+1)*tau when > 0

    @property
    def cap(self) -> int:
        if self.kv_cap:
            return self.kv_cap
        return self.kv_len_range[1] if self.kv_len_range else self.kv_len

    def layer_window(self, layer: int) -> int:
        if self.layer_pattern == "alternate" and layer % 2 == 0:
            return self.window
        return 0

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


SHAPE_TINY = LayerShape(hidden=256, n_q_heads=4, n_kv_heads=1, head_dim=64, n_experts=8,
                        top_k=2, n_local_experts=8, inter=256)
SHAPE_GPTOSS = LayerShape(hidden=2880, n_q_heads=64, n_kv_heads=8, head_dim=64, n_experts=128,
                          top_k=4, n_local_experts=4, inter=2880)

# the pages' own per-GPU slice: TP8 attention (8 query heads, 1 KV head per GPU), DP4 (512
# sequences per TP group), KV 32,768, RoPE; EP32 experts (4 local slots)
SHAPE_PAPER = LayerShape(hidden=2880, n_q_heads=8, n_kv_heads=1, head_dim=64, n_experts=128,
                         top_k=4, n_local_experts=4, inter=2880, rope_theta=150000.0)

WORKLOADS = {
    # tiny layer: 8 sequences, KV 128, 8 experts top-2, 2 microbatches of 4
    "tiny": Workload("tiny", SHAPE_TINY, n_tokens=8, n_layers=1, kv_len=128,
                     kv_sigma=1.0, microbatches=2),
    # one GPT-OSS-120B-shaped layer, per-GPU slice of a 32-GPU deployment
    "gptoss_layer": Workload("gptoss_layer", SHAPE_GPTOSS, n_tokens=64, n_layers=1,
                             kv_len=4096, microbatches=4),
    # 36-layer stack, alternating sliding-128 / full attention, KV 8192
    "gptoss_36l": Workload("gptoss_36l", SHAPE_GPTOSS, n_tokens=64, n_layers=36,
                           kv_len=8192, layer_pattern="alternate", microbatches=2),
    # the pages' decode configuration: 512 sequences x KV 32,768 per GPU, 36 layers
    "paper_32k": Workload("paper_32k", SHAPE_PAPER, n_tokens=512, n_layers=36,
                          kv_len=32768, layer_pattern="alternate", microbatches=2),
}


def sweep_workload(n_tokens: int, n_layers: int = 36) -> Workload:
    """Batch/length sweep point: ragged KV lengths uniform in [512, 16384]."""
    return Workload(f"sweep_b{n_tokens}", SHAPE_GPTOSS, n_tokens=n_tokens, n_layers=n_layers,
                    kv_len=16384, kv_len_range=(512, 16384), layer_pattern="alternate",
                    microbatches=2)


def skew_workload(n_layers: int = 36) -> Workload:
    """Skewed routing: Zipf(1.2)-shaped router bias with a block slot map."""
    shape = dataclasses.replace(SHAPE_GPTOSS, slot_map="block")
    return Workload("skew", shape, n_tokens=64, n_layers=n_layers, kv_len=8192,
                    layer_pattern="alternate", microbatches=2, zipf_bias=1.2)


# --------------------------------------------------------------------------
# tensor factories
# --------------------------------------------------------------------------
def x_in(wl: Workload, seed: int, device="cpu") -> torch.Tensor:
    return normal(seed, "x", 0, (wl.n_tokens, wl.shape.hidden), wl.x_sigma, device)


def kv_len(wl: Workload, seed: int, device="cpu") -> torch.Tensor:
    if wl.kv_len_range is None:
        return torch.full((wl.n_tokens,), wl.kv_len, dtype=torch.int32, device=device)
    lo, hi = wl.kv_len_range
    return uniform_int(seed, "kv_len", 0, wl.n_tokens, lo, hi, device)


def layer_weights(wl: Workload, layer: int, seed: int, device="cpu",
                  router_attempt: int = 0) -> dict:
    """Weights of one layer.  Matrices are row-major [out][in] (K-major rows)."""
    s = wl.shape
    ws = wl.w_sigma
    w = {
        "g_attn": normal(seed, "g_attn", layer, (s.hidden,), ws, device, mean_one=True),
        "w_qkv": normal(seed, "w_qkv", layer, (s.qkv_rows, s.hidden), ws, device),
        "w_o": normal(seed, "w_o", layer, (s.hidden, s.q_width), ws, device),
        "g_mlp": normal(seed, "g_mlp", layer, (s.hidden,), ws, device, mean_one=True),
        "w_router": normal(seed, f"w_router#{router_attempt}", layer, (s.n_experts, s.hidden),
                           ws, device),
        "w_gate_up": normal(seed, "w_gate_up", layer,
                            (s.n_local_experts, 2 * s.inter, s.hidden), ws, device),
        "w_down": normal(seed, "w_down", layer, (s.n_local_experts, s.hidden, s.inter),
                         ws, device),
        "router_bias": None,
    }
    if wl.zipf_bias > 0.0:
        g = torch.arange(s.n_experts, dtype=torch.float64)
        tau = ws * math.sqrt(s.hidden)          # scale of a router logit
        w["router_bias"] = (-wl.zipf_bias * tau * torch.log(g + 1.0)).to(torch.float32).to(device)
    return w


def kv_cache(wl: Workload, layer: int, seed: int, device="cpu"):
    """K and V caches bf16 [B][n_kv][cap][d]."""
    s = wl.shape
    shape = (wl.n_tokens, s.n_kv_heads, wl.cap, s.head_dim)
    return (normal(seed, "k_cache", layer, shape, wl.kv_sigma, device),
            normal(seed, "v_cache", layer, shape, wl.kv_sigma, device))


def kv_cache_rows(wl: Workload, layer: int, seed: int, seq: int, device="cpu"):
    """The K and V cache rows of one sequence, [n_kv][cap][d], equal to kv_cache()[seq]."""
    s = wl.shape
    per = s.n_kv_heads * wl.cap * s.head_dim
    shape = (s.n_kv_heads, wl.cap, s.head_dim)
    k = normal_flat(seed, "k_cache", layer, seq * per, per, wl.kv_sigma, device).view(*shape)
    v = normal_flat(seed, "v_cache", layer, seq * per, per, wl.kv_sigma, device).view(*shape)
    return k, v
