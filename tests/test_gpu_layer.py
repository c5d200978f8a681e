"""GPU parity of one decode layer (temporal execution) against the fp64 oracle,
through the C ABI.  Tolerance: max|err| <= 2e-2 * max|ref| per bf16 tensor;
routing sets bit-exact (inputs keep a top-k logit margin >= 1e-3)."""
import dataclasses

import numpy as np
import pytest
import torch

from intra_spatial_pipelining_gb300 import sgp, synth
from oracle import layer as O
from tests import harness as H

pytestmark = pytest.mark.gpu


def test_generator_identical_on_cpu_and_gpu():
    a = synth.normal(5, "k_cache", 3, (3, 5000), 0.02, "cpu")
    b = synth.normal(5, "k_cache", 3, (3, 5000), 0.02, "cuda").cpu()
    assert torch.equal(a, b)
    g1 = synth.normal(5, "g_attn", 1, (2880,), 0.02, "cpu", mean_one=True)
    g2 = synth.normal(5, "g_attn", 1, (2880,), 0.02, "cuda", mean_one=True).cpu()
    assert torch.equal(g1, g2)
    assert torch.equal(synth.kv_len(synth.sweep_workload(64, 1), 3, "cpu"),
                       synth.kv_len(synth.sweep_workload(64, 1), 3, "cuda").cpu())


def test_device_info():
    info = sgp.sgp_device_info_get()
    print(f"sm_count={info.sm_count} cc={info.cc_major}.{info.cc_minor} "
          f"green={info.green_ctx_supported} min_part={info.sm_min_partition} "
          f"align={info.sm_alignment} l2={info.l2_bytes}")
    assert info.sm_count > 0 and info.cc_major == 10


def _check_layer(inp, ref, res, T):
    s = inp.shape
    assert res["status"] == sgp.SGP_OK, sgp.sgp_status_string(res["status"])
    dmp = res["dump"]
    errs = {}
    for name in ("a", "q", "o", "h", "u"):
        errs[name] = H.assert_close(name, dmp[name], ref[name])
    ltol = 1e-3
    errs["logits"] = H.assert_close("logits", dmp["logits"], ref["logits"], tol=ltol)
    assert H.routing_sets(res["idx"]) == H.routing_sets(ref["idx"])
    # weights matched by expert index.  w = softmax over the selected logits, and
    # sum_i |dw_j/dz_i| = 2 w_j (1 - w_j) <= 1/2, so the logit bound above implies
    # |dw| <= ltol * max|z| / 2.
    wtol = 0.5 * ltol * float(np.abs(np.asarray(ref["logits"])).max())
    gi, gw = res["idx"].cpu().numpy(), res["w"].cpu().numpy()
    for t in range(T):
        g = dict(zip(gi[t].tolist(), gw[t].tolist()))
        for e, wv in zip(ref["idx"][t].tolist(), ref["w"][t].tolist()):
            assert abs(g[e] - wv) <= wtol, (t, e, g[e], wv, wtol)
    assert abs(float(gw.sum(axis=1).max()) - 1.0) < 1e-5
    # routed rows: slot order, pair positions
    off = dmp["slot_offsets"].cpu().numpy()
    pos = dmp["pair_pos"].cpu().numpy().reshape(T, s.top_k)
    slots = np.array([[O.slot_of(int(e), s.n_experts, s.n_local_experts, s.slot_map)
                       for e in row] for row in gi])
    for t in range(T):
        for j in range(s.top_k):
            assert off[slots[t, j]] <= pos[t, j] < off[slots[t, j] + 1]
    # dispatch is a stable counting sort of the pairs i = t k + j by slot: the slot sizes are
    # the counts, the positions are a permutation of the rows, and inside a slot the rows
    # follow the pair order (t, j)
    counts = np.bincount(slots.reshape(-1), minlength=s.n_local_experts)
    assert off[0] == 0 and np.array_equal(np.diff(off), counts)
    flat_pos, flat_slot = pos.reshape(-1), slots.reshape(-1)
    assert np.array_equal(np.sort(flat_pos), np.arange(T * s.top_k))
    for sl in range(s.n_local_experts):
        rows = flat_pos[flat_slot == sl]                  # in pair order i = t k + j
        assert np.array_equal(rows, np.arange(off[sl], off[sl + 1])), sl
    # SwiGLU rows and expert-down rows vs the oracle's per-pick values (matched by expert)
    zr = np.zeros((T * s.top_k, s.inter))
    yr = np.zeros((T * s.top_k, s.hidden))
    ri = ref["idx"]
    for t in range(T):
        for j in range(s.top_k):
            jr = list(ri[t]).index(gi[t, j])
            zr[pos[t, j]] = ref["z"][t][jr]
            yr[pos[t, j]] = ref["y"][t][jr]
    errs["z"] = H.assert_close("z", dmp["z"], zr)
    errs["y"] = H.assert_close("y", dmp["y"], yr)
    errs["x_next"] = H.assert_close("x_next", res["x_next"], ref["x_next"])
    return errs


@pytest.mark.parametrize("path", [sgp.PATH_GEMV, sgp.PATH_TC])
def test_tiny_layer_vs_oracle(path):
    wl = synth.WORKLOADS["tiny"]
    inp, ref = H.make_inputs_with_margin(wl, 1)
    res = H.run_temporal_layer(inp, H.dims(wl.shape, path))
    errs = _check_layer(inp, ref, res, wl.n_tokens)
    print("tiny", path, {k: f"{v:.2e}" for k, v in errs.items()})
    # the appended cache row equals the projection output
    k, v = inp.caches[0]
    L = inp.kv_len.cpu().numpy()
    kn = np.array([k[t, :, L[t] - 1].float().cpu().numpy().reshape(-1) for t in range(wl.n_tokens)])
    H.assert_close("k_new", kn, ref["k_new"].reshape(wl.n_tokens, -1))


@pytest.mark.parametrize("path", [sgp.PATH_AUTO, sgp.PATH_GEMV])
def test_gptoss_layer_vs_oracle(path):
    """Full C1 layer; forced onto the GEMV path it also covers several 16-token passes per
    matrix (64 tokens dense, about 64 routed rows per expert slot)."""
    wl = synth.WORKLOADS["gptoss_layer"]
    inp, ref = H.make_inputs_with_margin(wl, 2)
    res = H.run_temporal_layer(inp, H.dims(wl.shape, path))
    errs = _check_layer(inp, ref, res, wl.n_tokens)
    print("gptoss_layer", path, {k: f"{v:.2e}" for k, v in errs.items()})


@pytest.mark.parametrize("window", [0, 16, 200])
def test_ragged_lengths_and_windows(window):
    """Sequence lengths at MMA-tile (16), stage (64), half-chunk (512) and chunk (1024) edges."""
    wl = synth.WORKLOADS["tiny"].with_(n_tokens=12, kv_len=2400, kv_cap=2400)
    for a in range(20):
        inp = H.make_inputs(wl, 3, [a])
        inp.kv_len.copy_(torch.tensor([1, 17, 63, 64, 65, 511, 512, 513, 1023, 1024, 1025, 2300],
                                      dtype=torch.int32))
        # override the layer's window
        lay = inp.sgp_layers()[0]
        lay.window = window
        w = {n: (v.cpu() if v is not None else None) for n, v in inp.weights[0].items()}
        k, v = synth.kv_cache(wl, 0, inp.seed, "cpu")
        ref = O.layer(wl.shape, w, O.f64(inp.x), inp.kv_len.cpu().numpy(), O.f64(k), O.f64(v),
                      window)
        if min(O.topk_margin(z, wl.shape.top_k) for z in ref["logits"]) >= H.MARGIN:
            break
    d = H.dims(wl.shape, sgp.PATH_TC)
    ws = H.workspace(d, wl.n_tokens, wl.cap)
    out = torch.empty_like(inp.x)
    bufs, st = H.dump_buffers(wl.shape, wl.n_tokens)
    sgp.sgp_layer_temporal(d, lay, inp.kv_len, inp.x, out, wl.n_tokens, None, None, ws, st)
    assert sgp.sgp_status_from_workspace(ws) == sgp.SGP_OK
    H.assert_close("o", bufs["o"], ref["o"])
    H.assert_close("x_next", out, ref["x_next"])


@pytest.mark.parametrize("G", [1, 4, 8, 12, 16])
def test_attention_group_sizes(G):
    """Query heads per KV head from 1 to 16 (one or two head tiles, with padding heads)."""
    shape = dataclasses.replace(synth.SHAPE_TINY, n_q_heads=2 * G, n_kv_heads=2)
    wl = synth.WORKLOADS["tiny"].with_(shape=shape, n_tokens=6, kv_len=2200, kv_cap=2200)
    inp = H.make_inputs(wl, 5)
    inp.kv_len.copy_(torch.tensor([1, 100, 1024, 1500, 2049, 2200], dtype=torch.int32))
    lay = inp.sgp_layers()[0]
    w = {n: (v.cpu() if v is not None else None) for n, v in inp.weights[0].items()}
    k, v = synth.kv_cache(wl, 0, inp.seed, "cpu")
    ref = O.layer(wl.shape, w, O.f64(inp.x), inp.kv_len.cpu().numpy(), O.f64(k), O.f64(v), 0)
    d = H.dims(wl.shape, sgp.PATH_TC)
    ws = H.workspace(d, wl.n_tokens, wl.cap)
    out = torch.empty_like(inp.x)
    bufs, st = H.dump_buffers(wl.shape, wl.n_tokens)
    sgp.sgp_layer_temporal(d, lay, inp.kv_len, inp.x, out, wl.n_tokens, None, None, ws, st)
    assert sgp.sgp_status_from_workspace(ws) == sgp.SGP_OK
    H.assert_close("q", bufs["q"], ref["q"])
    H.assert_close("o", bufs["o"], ref["o"])


@pytest.mark.parametrize("path", [sgp.PATH_GEMV, sgp.PATH_TC])
def test_single_sequence_layer_vs_oracle(path):
    """One sequence: a single token row in every projection (one valid row of a 16-row MMA
    tile on the tensor-core path), one routed row per picked slot and empty slots elsewhere;
    a C1-shaped layer against the oracle on both projection paths."""
    wl = synth.WORKLOADS["gptoss_layer"].with_(n_tokens=1)
    inp, ref = H.make_inputs_with_margin(wl, 19)
    res = H.run_temporal_layer(inp, H.dims(wl.shape, path))
    errs = _check_layer(inp, ref, res, wl.n_tokens)
    print("one sequence", path, {k: f"{v:.2e}" for k, v in errs.items()})


@pytest.mark.parametrize("path", [sgp.PATH_GEMV, sgp.PATH_TC])
def test_largest_hidden_layer_vs_oracle(path):
    """hidden = 4096, the largest the library takes: the router's RMSNorm then loops over the
    row instead of holding it in registers, its shared-memory rows are at their widest, and
    the combine's fused next-layer RMSNorm keeps all 4096 features; every tensor against the
    oracle, on both projection paths."""
    shape = dataclasses.replace(synth.SHAPE_TINY, hidden=4096)
    wl = synth.WORKLOADS["tiny"].with_(shape=shape, n_tokens=24)
    inp, ref = H.make_inputs_with_margin(wl, 18)
    res = H.run_temporal_layer(inp, H.dims(wl.shape, path))
    errs = _check_layer(inp, ref, res, wl.n_tokens)
    print("hidden 4096", path, {k: f"{v:.2e}" for k, v in errs.items()})
    # a stack of two such layers: the combine also writes the next layer's RMSNorm input
    wl2 = wl.with_(n_layers=2)
    inp2, ref2 = H.make_stack_inputs_with_margin(wl2, 18)
    d = H.dims(wl2.shape, path)
    ws = H.workspace(d, wl2.n_tokens, wl2.cap)
    out = torch.empty_like(inp2.x)
    sgp.sgp_stack_temporal(d, inp2.sgp_layers(), inp2.kv_len, inp2.x, out, wl2.n_tokens,
                           None, None, ws)
    assert sgp.sgp_status_from_workspace(ws) == sgp.SGP_OK
    H.assert_close("x_out (2 layers)", out, ref2["x_out"])


def test_rope_layer_vs_oracle_long_positions():
    """RoPE on q and the new key (tensor-core QKV path) at positions up to 32,767."""
    shape = dataclasses.replace(synth.SHAPE_TINY, rope_theta=150000.0)
    wl = synth.WORKLOADS["tiny"].with_(shape=shape, n_tokens=16, kv_len=32768, kv_cap=32768)
    lens = [1, 2, 3, 64, 1000, 1023, 1024, 4096, 9999, 16384, 20000, 30000, 32000, 32766,
            32767, 32768]
    for a in range(20):
        inp = H.make_inputs(wl, 16, [a])
        inp.kv_len.copy_(torch.tensor(lens, dtype=torch.int32))
        w = {n: (v.cpu() if v is not None else None) for n, v in inp.weights[0].items()}
        k, v = synth.kv_cache(wl, 0, inp.seed, "cpu")
        ref = O.layer(wl.shape, w, O.f64(inp.x), inp.kv_len.cpu().numpy(), O.f64(k), O.f64(v), 0)
        if min(O.topk_margin(z, wl.shape.top_k) for z in ref["logits"]) >= H.MARGIN:
            break
    lay = inp.sgp_layers()[0]
    d = H.dims(wl.shape, sgp.PATH_TC)
    ws = H.workspace(d, wl.n_tokens, wl.cap)
    out = torch.empty_like(inp.x)
    bufs, st = H.dump_buffers(wl.shape, wl.n_tokens)
    sgp.sgp_layer_temporal(d, lay, inp.kv_len, inp.x, out, wl.n_tokens, None, None, ws, st)
    assert sgp.sgp_status_from_workspace(ws) == sgp.SGP_OK
    H.assert_close("q (rotated)", bufs["q"], ref["q"])
    kc = inp.caches[0][0]
    got_k = torch.stack([kc[t, :, lens[t] - 1] for t in range(wl.n_tokens)])
    H.assert_close("appended key (rotated)", got_k, ref["k_new"])
    H.assert_close("o", bufs["o"], ref["o"])
    H.assert_close("x_next", out, ref["x_next"])
    # RoPE needs the tensor-core QKV path
    with pytest.raises(sgp.SgpError) as e:
        sgp.sgp_layer_temporal(H.dims(wl.shape, sgp.PATH_GEMV), lay, inp.kv_len, inp.x, out,
                               wl.n_tokens, None, None, ws)
    assert e.value.code == sgp.SGP_ERR_INVALID_ARG


def test_invalid_arguments_are_rejected():
    wl = synth.WORKLOADS["tiny"]
    inp = H.make_inputs(wl, 4)
    d = H.dims(wl.shape)
    ws = H.workspace(d, wl.n_tokens, wl.cap)
    out = torch.empty_like(inp.x)
    lay = inp.sgp_layers()[0]
    bad = H.dims(wl.shape)
    bad.head_dim = 32
    with pytest.raises(sgp.SgpError) as e:
        sgp.sgp_layer_temporal(bad, lay, inp.kv_len, inp.x, out, wl.n_tokens, None, None, ws)
    assert e.value.code == sgp.SGP_ERR_INVALID_ARG
    small = ws[: ws.numel() // 2]
    with pytest.raises(sgp.SgpError) as e:
        sgp.sgp_layer_temporal(d, lay, inp.kv_len, inp.x, out, wl.n_tokens, None, None, small)
    assert e.value.code == sgp.SGP_ERR_INVALID_ARG


def test_out_of_range_kv_len_is_reported_not_faulted():
    wl = synth.WORKLOADS["tiny"]
    inp = H.make_inputs(wl, 5)
    inp.kv_len[3] = wl.cap + 7          # beyond the cache: kernels must skip and report
    res = H.run_temporal_layer(inp, H.dims(wl.shape), dump=False)
    assert res["status"] == sgp.SGP_ERR_DEVICE_BOUNDS
