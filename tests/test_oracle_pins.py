"""Pins of the fp64 oracle against facts that do not come from the oracle itself:
brute force on tiny inputs, closed forms, invariants, a library routine, and the
counts printed in "SubGPU Pipelining: Intra-GPU Fine-Grained Spatial Parallelism
for LLM Inference" (Section 4.2)."""
import dataclasses
import math
import os
import random

import numpy as np
import pytest
import torch

from oracle import layer as O
from oracle import schedule as S
from intra_spatial_pipelining_gb300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))


# ----------------------------------------------------------------------------- bf16
def test_bf16_matches_torch_on_fp32_values():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(200000) * np.exp(rng.uniform(-20, 20, 200000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(O.bf16(x.astype(np.float64)), ref)


def test_bf16_ties_to_even_and_exact_values():
    one = 1.0
    ulp = 2.0 ** -7
    assert O.bf16(one + ulp / 2) == one                    # tie -> even (1.0)
    assert O.bf16(one + 3 * ulp / 2) == one + 2 * ulp       # tie -> even mantissa
    assert O.bf16(one + ulp / 2 + 2.0 ** -30) == one + ulp  # above the tie rounds up
    assert O.bf16(-(one + ulp / 2)) == -one
    assert O.bf16(0.0) == 0.0
    assert O.bf16(3.0) == 3.0 and O.bf16(0.1) == 0.10009765625


# ----------------------------------------------------------------------------- rmsnorm
def test_rmsnorm_constant_vector_closed_form():
    g = np.linspace(0.5, 1.5, 32)
    c = -2.5
    y = O.rmsnorm(np.full(32, c), g, 1e-5)
    assert np.allclose(y, g * c / math.sqrt(c * c + 1e-5), rtol=1e-14, atol=0)


def test_rmsnorm_hand_example_and_scale_invariance():
    # x = (3, 4): mean(x^2) = 12.5
    y = O.rmsnorm(np.array([3.0, 4.0]), np.array([1.0, 2.0]), 0.0)
    assert np.allclose(y, [3 / math.sqrt(12.5), 8 / math.sqrt(12.5)], rtol=1e-15)
    x = np.random.default_rng(2).standard_normal(64)
    g = np.random.default_rng(3).standard_normal(64)
    assert np.allclose(O.rmsnorm(x, g, 0.0), O.rmsnorm(7.3 * x, g, 0.0), rtol=1e-13)


# ----------------------------------------------------------------------------- linear
def test_linear_brute_force():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((3, 5))
    w = rng.standard_normal((4, 5))
    y = O.linear(x, w)
    for t in range(3):
        for o in range(4):
            assert math.isclose(y[t, o], math.fsum(x[t, i] * w[o, i] for i in range(5)),
                                rel_tol=1e-13, abs_tol=1e-13)


# ----------------------------------------------------------------------------- attention
def _attention_brute(q, k, v, lo, hi):
    d = len(q)
    s = [sum(q[i] * k[p][i] for i in range(d)) / math.sqrt(d) for p in range(lo, hi)]
    mx = max(s)
    e = [math.exp(x - mx) for x in s]
    tot = math.fsum(e)
    return [math.fsum(e[j] * v[lo + j][i] for j in range(len(e))) / tot for i in range(d)]


@pytest.mark.parametrize("d,L,lo", [(4, 1, 0), (4, 9, 0), (8, 16, 5), (64, 12, 3)])
def test_attention_brute_force(d, L, lo):
    rng = np.random.default_rng(d * 100 + L)
    q, k, v = rng.standard_normal(d), rng.standard_normal((L, d)), rng.standard_normal((L, d))
    assert np.allclose(O.attention(q, k, v, lo, L), _attention_brute(q, k, v, lo, L),
                       rtol=1e-12, atol=1e-12)


def test_attention_identical_keys_give_mean_of_values():
    rng = np.random.default_rng(5)
    k = np.tile(rng.standard_normal(16), (40, 1))
    v = rng.standard_normal((40, 16))
    assert np.allclose(O.attention(rng.standard_normal(16), k, v, 7, 40),
                       v[7:40].mean(axis=0), rtol=1e-12, atol=1e-13)


def test_attention_single_position_and_dominant_logit():
    rng = np.random.default_rng(6)
    k, v = rng.standard_normal((10, 8)), rng.standard_normal((10, 8))
    assert np.allclose(O.attention(rng.standard_normal(8), k, v, 0, 1), v[0])
    q = np.ones(8)
    k2 = np.zeros((10, 8))
    k2[6] = 50.0                         # logit 400/sqrt(8) above all others
    assert np.allclose(O.attention(q, k2, v, 0, 10), v[6], atol=1e-12)


# ----------------------------------------------------------------------------- router
def test_topk_brute_force_sort_and_weights():
    rng = np.random.default_rng(7)
    for _ in range(50):
        z = rng.standard_normal(12)
        idx, w = O.topk(z, 3)
        full = sorted(range(12), key=lambda e: z[e], reverse=True)
        assert list(idx) == full[:3]
        assert math.isclose(float(np.sum(w)), 1.0, abs_tol=1e-12)
        # softmax over the selection == full softmax renormalised over the selection
        pf = np.exp(z - z.max())
        pf = pf / pf.sum()
        assert np.allclose(w, pf[idx] / pf[idx].sum(), rtol=1e-12)
        assert np.all(np.diff(z[idx]) <= 0)


def test_topk_ties_go_to_lower_index_and_margin():
    z = np.array([1.0, 3.0, 2.0, 3.0, 2.0])
    idx, w = O.topk(z, 3)
    assert list(idx) == [1, 3, 2]
    assert O.topk_margin(z, 2) == 1.0 and O.topk_margin(z, 3) == 0.0
    assert np.allclose(w[:2], w[0]) and w[0] > w[2]


def test_slot_maps():
    assert [O.slot_of(g, 8, 4, "mod") for g in range(8)] == [0, 1, 2, 3, 0, 1, 2, 3]
    assert [O.slot_of(g, 8, 4, "block") for g in range(8)] == [0, 0, 1, 1, 2, 2, 3, 3]
    assert [O.slot_of(g, 8, 8, "mod") for g in range(8)] == list(range(8))


# ----------------------------------------------------------------------------- experts
def test_silu_closed_forms():
    assert O.silu(np.array(0.0)) == 0.0
    assert math.isclose(float(O.silu(np.array(1.0))), 1.0 / (1.0 + math.exp(-1.0)), rel_tol=1e-15)
    assert math.isclose(float(O.silu(np.array(40.0))), 40.0, rel_tol=1e-15)
    assert abs(float(O.silu(np.array(-40.0)))) < 1e-15


def test_swiglu_expert_brute_force():
    rng = np.random.default_rng(8)
    H, I = 6, 4
    u = rng.standard_normal(H)
    wgu = rng.standard_normal((2 * I, H))
    wd = rng.standard_normal((H, I))
    z, y = O.swiglu_expert(u, wgu, wd, I)
    zb = []
    for i in range(I):
        g = math.fsum(wgu[i, c] * u[c] for c in range(H))
        up = math.fsum(wgu[I + i, c] * u[c] for c in range(H))
        zb.append(float(O.bf16(g / (1 + math.exp(-g)) * up)))
    assert np.array_equal(z, zb)
    for c in range(H):
        assert math.isclose(y[c], math.fsum(wd[c, i] * zb[i] for i in range(I)),
                            rel_tol=1e-12, abs_tol=1e-12)


# ----------------------------------------------------------------------------- whole layer
TINY = synth.LayerShape(hidden=16, n_q_heads=4, n_kv_heads=2, head_dim=4, n_experts=4,
                        top_k=2, n_local_experts=4, inter=8)


def _np_weights(shape, seed, zero=()):
    wl = synth.Workload("t", shape, n_tokens=3, n_layers=1, kv_len=6, kv_sigma=1.0, w_sigma=0.3)
    w = synth.layer_weights(wl, 0, seed)
    out = {n: (O.f64(v) if v is not None else None) for n, v in w.items()}
    for n in zero:
        out[n] = np.zeros_like(out[n])
    return wl, out


def _caches(wl, seed):
    k, v = synth.kv_cache(wl, 0, seed)
    return O.f64(k).copy(), O.f64(v).copy()


def test_layer_brute_force_tiny():
    """Whole layer vs a loop-by-loop evaluation of its definition on a tiny shape."""
    wl, W = _np_weights(TINY, 11)
    kc, vc = _caches(wl, 11)
    x = O.f64(synth.x_in(wl, 11))
    kvl = np.array([6, 3, 1])
    r = O.layer(TINY, W, x, kvl, kc.copy(), vc.copy(), window=0)
    s = TINY
    for t in range(3):
        xt = list(x[t])
        ms = math.fsum(v * v for v in xt) / s.hidden
        a = [float(O.bf16(xt[c] / math.sqrt(ms + s.rms_eps) * W["g_attn"][c])) for c in range(s.hidden)]
        qkv = [math.fsum(W["w_qkv"][o][c] * a[c] for c in range(s.hidden)) for o in range(s.qkv_rows)]
        qkv = [float(O.bf16(v)) for v in qkv]
        L = int(kvl[t])
        K = [[list(kc[t, h, p]) for p in range(L)] for h in range(2)]
        V = [[list(vc[t, h, p]) for p in range(L)] for h in range(2)]
        for h in range(2):
            K[h][L - 1] = qkv[16 + 4 * h:16 + 4 * h + 4]
            V[h][L - 1] = qkv[24 + 4 * h:24 + 4 * h + 4]
        o = []
        for h in range(4):
            o += _attention_brute(qkv[4 * h:4 * h + 4], K[h // 2], V[h // 2], 0, L)
        o = [float(O.bf16(v)) for v in o]
        hr = [float(O.bf16(xt[c] + math.fsum(W["w_o"][c][i] * o[i] for i in range(16))))
              for c in range(16)]
        ms = math.fsum(v * v for v in hr) / 16
        u = [float(O.bf16(hr[c] / math.sqrt(ms + s.rms_eps) * W["g_mlp"][c])) for c in range(16)]
        z = [math.fsum(W["w_router"][e][c] * u[c] for c in range(16)) for e in range(4)]
        top = sorted(range(4), key=lambda e: (-z[e], e))[:2]
        ez = [math.exp(z[e] - z[top[0]]) for e in top]
        wt = [v / math.fsum(ez) for v in ez]
        acc = [0.0] * 16
        for j, e in enumerate(top):
            g = [math.fsum(W["w_gate_up"][e][i][c] * u[c] for c in range(16)) for i in range(8)]
            up = [math.fsum(W["w_gate_up"][e][8 + i][c] * u[c] for c in range(16)) for i in range(8)]
            zz = [float(O.bf16(g[i] / (1 + math.exp(-g[i])) * up[i])) for i in range(8)]
            for c in range(16):
                acc[c] += wt[j] * math.fsum(W["w_down"][e][c][i] * zz[i] for i in range(8))
        xn = [float(O.bf16(hr[c] + acc[c])) for c in range(16)]
        assert list(r["idx"][t]) == top
        assert np.allclose(r["w"][t], wt, rtol=1e-12)
        for name, ref in (("a", a), ("o", o), ("h", hr), ("u", u)):
            assert np.array_equal(r[name][t], ref), name
        assert np.allclose(r["x_next"][t], xn, rtol=0, atol=2 ** -6 * max(1.0, max(map(abs, xn))))


def test_layer_gqa_mapping_and_window():
    """q = k_new = v_new = 0 (zero QKV weights), so every score is 0 and each
    query head outputs the mean of its KV head's V rows over the window.  Each KV
    head holds a different constant V, and positions before the window are
    poisoned: a wrong head mapping or a wrong window start changes the output."""
    wl, W = _np_weights(TINY, 12, zero=("w_qkv",))
    kc, vc = _caches(wl, 12)
    kvl = np.array([6, 6, 6])
    for h in range(2):
        vc[:, h] = 1.0 + h
    vc[:, :, :2] = 1e6                   # before the window [L-4, L)
    x = O.f64(synth.x_in(wl, 12))
    r = O.layer(TINY, W, x, kvl, kc, vc, window=4)
    o = r["o"].reshape(3, 4, 4)
    # window [2, 6): three rows of value (1 + kv_head) and the appended zero row
    for h in range(4):
        assert np.all(o[:, h] == 3 * (1.0 + h // 2) / 4.0)
    assert np.all(kc[:, :, 5] == 0.0) and np.all(vc[:, :, 5] == 0.0)
    assert np.all(vc[:, :, 4] == vc[:, :, 3])


def test_layer_zero_weights_are_residual_only():
    wl, W = _np_weights(TINY, 13, zero=("w_o", "w_down"))
    kc, vc = _caches(wl, 13)
    x = O.f64(synth.x_in(wl, 13))
    r = O.layer(TINY, W, x, np.array([6, 5, 4]), kc, vc, window=0)
    assert np.array_equal(r["h"], x)       # x is already on the bf16 grid
    assert np.array_equal(r["x_next"], x)


def test_layer_identical_experts_weights_sum_to_one():
    """All slots hold the same expert: the combine must add exactly one expert
    output (the weights sum to 1), whatever the routing."""
    wl, W = _np_weights(TINY, 14)
    W["w_gate_up"][:] = W["w_gate_up"][0]
    W["w_down"][:] = W["w_down"][0]
    kc, vc = _caches(wl, 14)
    x = O.f64(synth.x_in(wl, 14))
    r = O.layer(TINY, W, x, np.array([6, 5, 4]), kc, vc, window=0)
    for t in range(3):
        _, y = O.swiglu_expert(r["u"][t], W["w_gate_up"][0], W["w_down"][0], TINY.inter)
        ref = r["h"][t] + y
        # equal up to fp64 rounding of sum_j w_j*y before the bf16 rounding
        assert np.max(np.abs(r["x_next"][t] - O.bf16(ref))) <= 2.0 ** -8 * np.max(np.abs(ref))
        assert np.mean(r["x_next"][t] == O.bf16(ref)) > 0.9


def test_layer_router_bias_forces_selection_and_mod_slots():
    shape = dataclasses.replace(TINY, n_experts=8, n_local_experts=4)
    wl, W = _np_weights(shape, 15)
    W["router_bias"] = np.zeros(8)
    W["router_bias"][6] = 1e3
    kc, vc = _caches(wl, 15)
    x = O.f64(synth.x_in(wl, 15))
    r = O.layer(shape, W, x, np.array([6, 5, 4]), kc, vc, window=0)
    assert np.all(r["idx"][:, 0] == 6) and np.all(r["slot"][:, 0] == 2)
    assert np.allclose(r["w"][:, 0], 1.0) and np.all(r["w"][:, 1] < 1e-12)


def test_layer_dense_mlp_special_case():
    """One expert, top-1: the MoE reduces to a dense SwiGLU MLP with weight 1."""
    shape = dataclasses.replace(TINY, n_experts=1, top_k=1, n_local_experts=1)
    wl, W = _np_weights(shape, 16)
    kc, vc = _caches(wl, 16)
    x = O.f64(synth.x_in(wl, 16))
    r = O.layer(shape, W, x, np.array([6, 5, 4]), kc, vc, window=0)
    for t in range(3):
        u = r["u"][t]
        g = W["w_gate_up"][0][:8] @ u
        up = W["w_gate_up"][0][8:] @ u
        mlp = W["w_down"][0] @ O.bf16(g * (1 / (1 + np.exp(-g))) * up)
        assert np.allclose(r["x_next"][t], O.bf16(r["h"][t] + mlp), rtol=0, atol=1e-12)
        assert r["w"][t][0] == 1.0


def test_layer_is_per_token_and_idempotent():
    """Microbatching does not change results (each token's output depends only
    on its own row and its own sequence's cache), and re-running rewrites the
    same cache slot with the same values."""
    wl, W = _np_weights(TINY, 17)
    kc, vc = _caches(wl, 17)
    x = O.f64(synth.x_in(wl, 17))
    kvl = np.array([6, 2, 5])
    full = O.layer(TINY, W, x, kvl, kc.copy(), vc.copy(), window=3)
    k2, v2 = kc.copy(), vc.copy()
    parts = [O.layer(TINY, W, x, kvl, k2, v2, window=3, tokens=[t]) for t in (2, 0, 1)]
    again = O.layer(TINY, W, x, kvl, k2, v2, window=3)
    for t, p in zip((2, 0, 1), parts):
        assert np.array_equal(p["x_next"][0], full["x_next"][t])
    assert np.array_equal(again["x_next"], full["x_next"])


# ----------------------------------------------------------------------------- schedule
def _golden_counts():
    rows = {}
    with open(os.path.join(HERE, "golden", "search_space_counts.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                name, n, st, qu, cnt = line.split()
                rows[name] = (int(n), int(st), int(qu), int(cnt))
    return rows


def test_search_space_counts_printed_on_the_page():
    g = _golden_counts()
    n, st, _, cnt = g["cut_and_binding_choices_20_operator_chain"]
    assert S.count_cut_bindings(n, st) == cnt
    n, st, qu, cnt = g["sm_allocations_148_sms_2sm_quantum"]
    assert S.count_allocations_closed(n, st, qu) == cnt
    assert S.count_allocations(n, st, qu) == cnt


def test_binding_eq1():
    assert [S.binding(k, 3, 0) for k in (1, 2, 3)] == [1, 2, 3]
    assert [S.binding(k, 3, 1) for k in (1, 2, 3)] == [1, 2, 1]


def test_makespan_hand_example():
    # 1 layer, 2 microbatches, 2 segments: tau_A = 3, tau_B = 2
    tasks = S.build_tasks(1, 2, 2)
    T, A, C = S.makespan(tasks, [3, 2, 3, 2])
    assert (A, C, T) == ([0, 3, 3, 6], [3, 5, 6, 8], 8)


def test_makespan_two_stage_closed_form():
    # one layer, m microbatches, two stages: fill + (m-1) * slowest + drain
    for ta, tb in ((3.0, 2.0), (1.0, 4.0), (2.5, 2.5)):
        for m in (1, 2, 5, 9):
            tasks = S.build_tasks(1, m, 2)
            tau = [ta if t["seg"] == 1 else tb for t in tasks]
            T, _, _ = S.makespan(tasks, tau)
            assert math.isclose(T, ta + tb + (m - 1) * max(ta, tb))


def test_makespan_equals_longest_path_random():
    rnd = random.Random(3)
    for _ in range(30):
        L, m, K = rnd.randint(1, 4), rnd.randint(1, 4), rnd.randint(2, 4)
        w = rnd.randint(0, 1) if K > 2 else 0
        tasks = S.build_tasks(L, m, K, w)
        tau = [rnd.uniform(0.1, 3.0) for _ in tasks]
        assert math.isclose(S.makespan(tasks, tau)[0], S.longest_path(tasks, tau))
        # stage edges serialise each stage: no two tasks on a stage overlap
        _, A, C = S.makespan(tasks, tau)
        for st in {t["stage"] for t in tasks}:
            iv = sorted((A[t["id"]], C[t["id"]]) for t in tasks if t["stage"] == st)
            assert all(iv[i][1] <= iv[i + 1][0] + 1e-12 for i in range(len(iv) - 1))


# ---------------------------------------------------------------------------
# RoPE (half-split pairs), pinned by properties of rotations and by the complex form
# ---------------------------------------------------------------------------
def test_rope_position_zero_is_identity_and_norm_is_kept():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((3, 64))
    assert np.array_equal(O.rope(x, 0, 150000.0), x)
    y = O.rope(x, 12345, 150000.0)
    assert np.allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)


def test_rope_scores_depend_on_relative_position_only():
    rng = np.random.default_rng(12)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    s1 = O.rope(q, 5, 10000.0) @ O.rope(k, 2, 10000.0)
    s2 = O.rope(q, 30003, 10000.0) @ O.rope(k, 30000, 10000.0)
    assert abs(s1 - s2) < 1e-9 * max(1.0, abs(s1))
    # and composition adds positions
    x = rng.standard_normal(64)
    assert np.allclose(O.rope(O.rope(x, 7, 500.0), 11, 500.0), O.rope(x, 18, 500.0), atol=1e-12)


def test_rope_matches_complex_rotation():
    """Pair i (x_i, x_{i+d/2}) is the complex number x_i + j x_{i+d/2} times e^{j pos w_i},
    w_i = theta^(-2i/d): a second formulation of the same rotation."""
    rng = np.random.default_rng(13)
    d, pos, theta = 8, 3, 100.0
    x = rng.standard_normal(d)
    zc = (x[: d // 2] + 1j * x[d // 2:]) * np.exp(1j * pos * theta ** (-np.arange(0, d, 2) / d))
    assert np.allclose(O.rope(x, pos, theta), np.concatenate([zc.real, zc.imag]), atol=1e-13)


def test_layer_rope_rotates_q_and_new_key_only():
    """With RoPE on, q and the appended key are the unrotated ones rotated at L-1; the
    appended value is untouched (tiny layer, brute-force comparison with RoPE off)."""
    import dataclasses
    wl = synth.WORKLOADS["tiny"].with_(n_tokens=3, kv_len=40)
    w = synth.layer_weights(wl, 0, 21, "cpu")
    x = O.f64(synth.x_in(wl, 21))
    kvl = np.array([1, 17, 40])
    k, v = synth.kv_cache(wl, 0, 21, "cpu")
    plain = O.layer(wl.shape, w, x, kvl, O.f64(k), O.f64(v), 0)
    shape_r = dataclasses.replace(wl.shape, rope_theta=10000.0)
    rot = O.layer(shape_r, w, x, kvl, O.f64(k), O.f64(v), 0)
    nq, d = wl.shape.n_q_heads, wl.shape.head_dim
    for i, L in enumerate(kvl):
        # rounding happens after the rotation: compare through the unrounded projection
        a = plain["a"][i]
        qkv = O.linear(a, O.f64(w["w_qkv"]))
        q_ref = O.bf16(O.rope(qkv[: nq * d].reshape(nq, d), int(L) - 1, 10000.0)).reshape(-1)
        assert np.array_equal(rot["q"][i], q_ref)
        assert np.array_equal(rot["v_new"][i], plain["v_new"][i])
    assert np.array_equal(rot["q"][0], plain["q"][0])   # L = 1: position 0, no rotation


def test_rope_frequencies_written_out_by_hand():
    """RoFormer's schedule theta_i = theta^(-2(i-1)/d), i = 1..d/2, written out by hand:
    d = 4, theta = 100 gives angular rates {1, 0.1}; d = 8, theta = 10000 gives
    {1, 0.1, 0.01, 0.001}.  Pair i is (x_i, x_{i+d/2}) (half-split).  A schedule
    theta^(-i/d) or a transposed pairing fails here."""
    x = np.array([1.0, 2.0, 3.0, 4.0])
    c1, s1, c01, s01 = math.cos(1.0), math.sin(1.0), math.cos(0.1), math.sin(0.1)
    want = [1 * c1 - 3 * s1, 2 * c01 - 4 * s01, 1 * s1 + 3 * c1, 2 * s01 + 4 * c01]
    assert np.allclose(O.rope(x, 1, 100.0), want, rtol=0, atol=1e-15)
    # position 2 doubles every angle
    c2, s2, c02, s02 = math.cos(2.0), math.sin(2.0), math.cos(0.2), math.sin(0.2)
    want = [1 * c2 - 3 * s2, 2 * c02 - 4 * s02, 1 * s2 + 3 * c2, 2 * s02 + 4 * c02]
    assert np.allclose(O.rope(x, 2, 100.0), want, rtol=0, atol=1e-15)
    # d = 8: unit vectors in the first half pick out (cos, sin) of each rate
    for i, rate in enumerate((1.0, 0.1, 0.01, 0.001)):
        e = np.zeros(8)
        e[i] = 1.0
        y = O.rope(e, 1, 10000.0)
        assert math.isclose(y[i], math.cos(rate), rel_tol=0, abs_tol=1e-15)
        assert math.isclose(y[i + 4], math.sin(rate), rel_tol=0, abs_tol=1e-15)
        assert np.count_nonzero(y) == 2


# ---------------------------------------------------------------------------
# the stack: layer l's output feeds layer l+1, each layer with its own cache
# ---------------------------------------------------------------------------
def test_stack_equals_layers_chained_by_hand():
    """Three layers with windows [2, 0, 4], a separate cache per layer and the token
    subset [2, 0] (out of order).  The reference chains the pinned one-layer oracle by hand,
    token by token, each layer on its own copy of its own cache.  A wrong cache per layer,
    a wrong window, or a row scattered to the wrong token changes the result."""
    wl = synth.Workload("t", TINY, n_tokens=3, n_layers=3, kv_len=6, kv_sigma=1.0, w_sigma=0.3)
    seed = 31
    weights = [{n: (O.f64(v) if v is not None else None)
                for n, v in synth.layer_weights(wl, l, seed).items()} for l in range(3)]
    caches = []
    for l in range(3):
        k, v = synth.kv_cache(wl, l, seed)
        caches.append((O.f64(k).copy(), O.f64(v).copy()))
    x = O.f64(synth.x_in(wl, seed))
    kvl = np.array([6, 4, 5])
    windows = [2, 0, 4]
    tokens = [2, 0]
    ref_caches = [(k.copy(), v.copy()) for k, v in caches]
    untouched = [(k.copy(), v.copy()) for k, v in caches]
    r = O.stack(TINY, weights, windows, x, kvl, caches, tokens=tokens)

    for i, t in enumerate(tokens):
        cur = x.copy()
        for l in range(3):
            one = O.layer(TINY, weights[l], cur, kvl, ref_caches[l][0], ref_caches[l][1],
                          windows[l], tokens=[t])
            cur = cur.copy()
            cur[t] = one["x_next"][0]
            assert np.array_equal(r["idx"][l][i], one["idx"][0])
            assert np.array_equal(r["w"][l][i], one["w"][0])
            assert np.array_equal(r["logits"][l][i], one["logits"][0])
        assert np.array_equal(r["x_out"][i], cur[t])
    # every layer's cache received its own appended rows, and only the listed tokens'
    for l in range(3):
        assert np.array_equal(caches[l][0], ref_caches[l][0])
        assert np.array_equal(caches[l][1], ref_caches[l][1])
        assert np.array_equal(caches[l][0][1], untouched[l][0][1])
        for t in tokens:
            assert not np.array_equal(caches[l][0][t, :, kvl[t] - 1], untouched[l][0][t, :, kvl[t] - 1])
    # the layers differ from each other, so a shared cache or weight set would be visible
    assert not np.array_equal(r["idx"][0], r["idx"][1]) or not np.array_equal(r["w"][0], r["w"][1])


def test_steady_state_period_is_the_growth_rate_of_the_makespan():
    """Each extra microbatch adds the slowest stage's time to the Eq. 4-5 makespan of a
    chain pipeline: the steady-state period is max_d tau_d."""
    rnd = random.Random(5)
    for _ in range(20):
        K = rnd.randint(2, 4)
        tau_st = [rnd.uniform(0.2, 3.0) for _ in range(K)]
        spans = []
        for m in (6, 7):
            tasks = S.build_tasks(1, m, K)
            spans.append(S.makespan(tasks, [tau_st[t["seg"] - 1] for t in tasks])[0])
        assert math.isclose(spans[1] - spans[0], S.steady_state_period(tau_st), rel_tol=1e-12)


def test_two_lanes_per_stage_hand_example():
    """Two FIFOs per stage (microbatch parity): one layer, 2 microbatches, 2 segments,
    tau_A = 3, tau_B = 2.  With one lane microbatch 1's stage-A task waits for microbatch 0's
    (it starts at 3); with two lanes it starts at 0, and both finish at 5 -- the model then
    assumes the pool fits both tasks at full speed, a bound the measurement checks."""
    one = S.build_tasks(1, 2, 2)
    two = S.build_tasks(1, 2, 2, lanes=2)
    assert S.makespan(one, [3, 2, 3, 2])[0] == 8
    T, A, C = S.makespan(two, [3, 2, 3, 2])
    assert (A, C, T) == ([0, 3, 0, 3], [3, 5, 3, 5], 5)
    assert [t["stage_pred"] for t in two] == [None, None, None, None]
    four = S.build_tasks(1, 4, 2, lanes=2)
    assert [t["stage_pred"] for t in four] == [None, None, None, None, 0, 1, 2, 3]
