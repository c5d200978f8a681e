"""The seeded generator: determinism, slicing, moments (no layer arithmetic here)."""
import torch

from intra_spatial_pipelining_gb300 import synth


def test_deterministic_and_key_separated():
    a = synth.normal(7, "w_o", 3, (64, 40), 0.02)
    b = synth.normal(7, "w_o", 3, (64, 40), 0.02)
    c = synth.normal(7, "w_o", 4, (64, 40), 0.02)
    d = synth.normal(8, "w_o", 3, (64, 40), 0.02)
    assert a.dtype == torch.bfloat16 and torch.equal(a, b)
    assert not torch.equal(a, c) and not torch.equal(a, d)


def test_moments_and_bounds():
    v = synth.normal(1, "x", 0, (1 << 20,), 1.0).float()
    assert abs(v.mean().item()) < 3e-3
    assert abs(v.std().item() - 1.0) < 3e-3
    assert v.abs().max().item() < 3.47
    g = synth.normal(1, "g", 0, (1 << 16,), 0.02, mean_one=True).float()
    assert abs(g.mean().item() - 1.0) < 1e-3 and abs(g.std().item() - 0.02) < 1e-3


def test_sequence_slice_equals_full_cache():
    wl = synth.WORKLOADS["tiny"].with_(n_tokens=5, kv_len=40)
    k, v = synth.kv_cache(wl, 2, 9)
    for seq in (0, 3, 4):
        ks, vs = synth.kv_cache_rows(wl, 2, 9, seq)
        assert torch.equal(ks, k[seq]) and torch.equal(vs, v[seq])


def test_chunked_generation_matches_unchunked(monkeypatch):
    ref = synth.normal(3, "k_cache", 1, (3000,), 0.5)
    monkeypatch.setattr(synth, "_CHUNK", 257)
    assert torch.equal(synth.normal(3, "k_cache", 1, (3000,), 0.5), ref)


def test_ragged_lengths_in_range():
    wl = synth.sweep_workload(256, n_layers=1)
    L = synth.kv_len(wl, 5)
    assert L.dtype == torch.int32 and L.min().item() >= 512 and L.max().item() <= 16384
    assert len(set(L.tolist())) > 200
    assert wl.cap == 16384


def test_workload_shapes():
    wl = synth.WORKLOADS["gptoss_36l"]
    assert [wl.layer_window(l) for l in range(4)] == [128, 0, 128, 0]
    w = synth.layer_weights(synth.WORKLOADS["tiny"], 0, 1)
    s = synth.SHAPE_TINY
    assert w["w_qkv"].shape == (s.qkv_rows, s.hidden)
    assert w["w_gate_up"].shape == (s.n_local_experts, 2 * s.inter, s.hidden)
    assert w["w_down"].shape == (s.n_local_experts, s.hidden, s.inter)
