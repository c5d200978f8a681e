"""Pairwise-line SM-allocation refinement ("SubGPU Pipelining: Intra-GPU Fine-Grained
Spatial Parallelism for LLM Inference", Section 4.2, Algorithm 2).

The schedule model's restatement of the algorithm is pinned against brute force over every
legal allocation for objectives where a pairwise search must find the optimum (the maximum
of per-stage times that fall as a stage gets SMs); the library's C implementation is then
checked step for step against the model on arbitrary objectives (same allocation, same
value, same set of evaluated allocations)."""
import math
import random

import pytest

from intra_spatial_pipelining_gb300 import build, sgp
from oracle import schedule as S


@pytest.fixture(scope="module")
def lib():
    build.build()
    return sgp.lib()


def _uniform_seed(n_sm, n, g):
    q = n_sm // g
    p = [(q // n) * g] * n
    p[-1] += n_sm - sum(p)
    return tuple(p)


def _stage_time_objective(w, c):
    """max_d (w_d / p_d + c_d): a stage's time falls as it gets SMs; the slowest stage sets
    the steady-state period."""
    return lambda p: max(wi / pi + ci for wi, pi, ci in zip(w, p, c))


@pytest.mark.parametrize("n_stages", [2, 3, 4])
def test_model_reaches_the_brute_force_optimum_on_stage_time_objectives(n_stages):
    rnd = random.Random(40 + n_stages)
    n_sm, g, p_min = 152, 8, 8
    feas = lambda p: min(p) >= max(p_min, g)
    for _ in range(15):
        w = [rnd.uniform(0.5, 8.0) for _ in range(n_stages)]
        c = [rnd.uniform(0.0, 0.05) for _ in range(n_stages)]
        f = _stage_time_objective(w, c)
        best = min(f(p) for p in S.allocations(n_sm, n_stages, g, p_min))
        for seed in (_uniform_seed(n_sm, n_stages, g),
                     tuple([p_min] * (n_stages - 1) + [n_sm - p_min * (n_stages - 1)])):
            p, t = S.pairwise_line(f, feas, seed, g)
            assert feas(p) and sum(p) == n_sm
            assert math.isclose(t, f(p)) and math.isclose(t, best, rel_tol=1e-12), (w, seed, p)


def test_model_line_search_doubles_then_halves():
    """Hand example, one pass, quantum 1 SM: f = 1.001 |p_1 - 40| on the line p_0 + p_1 = 112,
    start (104, 8).  The one-quantum moves are (103, 9) and (105, 7); the first improves, so the
    line search steps z = 2, 4, 8, 16, 32 (each better), 64 (worse: h halves), 48, 40, 36, 34,
    33 (all worse than z = 32) and keeps z = 32, i.e. (72, 40)."""
    f = lambda p: abs(p[1] - 40) + abs(p[0] - 72) * 1e-3
    seen = []

    def rec(p):
        if p not in seen:
            seen.append(p)
        return f(p)
    p, t = S.pairwise_line(rec, lambda p: min(p) >= 1, (104, 8), 1, passes=1)
    assert p == (72, 40) and t == 0.0
    line = [(104 - z, 8 + z) for z in (2, 4, 8, 16, 32, 64, 48, 40, 36, 34, 33)]
    assert seen == [(104, 8), (103, 9), (105, 7)] + line


def _random_table(seed):
    rnd = random.Random(seed)
    cache = {}

    def f(p):
        if p not in cache:
            cache[p] = rnd.random() if rnd.random() > 0.05 else -1.0   # some cannot be evaluated
        return cache[p]
    return f


@pytest.mark.parametrize("n_stages", [2, 3, 4])
def test_library_follows_the_model_step_for_step(lib, n_stages):
    n_sm, g, p_min = 152, 8, 16
    feas = lambda p: min(p) >= max(p_min, g)
    for trial in range(25):
        table = _random_table(1000 * n_stages + trial)
        f_model = lambda p: (lambda v: math.inf if v < 0 else v)(table(p))
        seen_model, seen_lib = set(), set()

        def fm(p):
            seen_model.add(p)
            return f_model(p)

        def fl(p):
            seen_lib.add(p)
            return table(p)
        seed = _uniform_seed(n_sm, n_stages, g)
        limit = 0 if trial % 2 else 3
        pm, tm = S.pairwise_line(fm, feas, seed, g, passes=limit or None)
        pl, tl, n_eval = sgp.sgp_refine_allocation(seed, g, p_min, fl, pass_limit=limit)
        assert pl == pm and (tl == tm or (math.isinf(tl) and math.isinf(tm)))
        assert seen_lib == seen_model and n_eval == len(seen_lib)


def test_library_on_stage_time_objectives_matches_brute_force(lib):
    rnd = random.Random(7)
    for _ in range(10):
        w = [rnd.uniform(0.5, 8.0) for _ in range(3)]
        f = _stage_time_objective(w, [0.0, 0.0, 0.0])
        best = min(f(p) for p in S.allocations(152, 3, 8, 8))
        p, t, n_eval = sgp.sgp_refine_allocation((48, 48, 56), 8, 8, f)
        assert math.isclose(t, best, rel_tol=1e-12) and sum(p) == 152
        assert n_eval < sum(1 for _ in S.allocations(152, 3, 8, 8))


def test_library_refuses_bad_arguments(lib):
    with pytest.raises(sgp.SgpError):
        sgp.sgp_refine_allocation((152,), 8, 8, lambda p: 1.0)          # one stage
    with pytest.raises(sgp.SgpError):
        sgp.sgp_refine_allocation((4, 148), 8, 8, lambda p: 1.0)        # below p_min


# ----------------------------------------------------------------------------- Eq. 4-5
def _model_arrays(tasks):
    return ([t["data"][0] if t["data"] else -1 for t in tasks],
            [t["stage_pred"] if t["stage_pred"] is not None else -1 for t in tasks],
            [t["stage"] for t in tasks])


def test_library_makespan_equals_the_schedule_model(lib):
    """The recurrence the makespan predictor runs equals the schedule model's Eq. 4-5 (no
    handoff) on random DAGs of 1-4 layers, 1-4 microbatches, 2-4 segments, with and without
    boundary reuse and with one or two lanes per stage."""
    rnd = random.Random(9)
    for _ in range(40):
        L, m, K = rnd.randint(1, 4), rnd.randint(1, 4), rnd.randint(2, 4)
        w = rnd.randint(0, 1) if K > 2 else 0
        tasks = S.build_tasks(L, m, K, w, lanes=rnd.choice([1, 2]))
        tau = [rnd.uniform(0.1, 3.0) for _ in tasks]
        pd, ps, st = _model_arrays(tasks)
        T, fin = sgp.sgp_makespan(pd, ps, st, tau)
        T_model, _, C_model = S.makespan(tasks, tau)
        assert math.isclose(T, T_model, rel_tol=1e-12)
        assert all(math.isclose(a, b, rel_tol=1e-12) for a, b in zip(fin, C_model))


def test_library_makespan_handoff_hand_example(lib):
    """One layer, 2 microbatches, 2 stages, tau_A = 3, tau_B = 2, handoff 1 on the A -> B edges:
    A0 [0, 3], B0 [4, 6], A1 [3, 6], B1 [7, 9] -> 9 (8 without the handoff)."""
    tasks = S.build_tasks(1, 2, 2)
    pd, ps, st = _model_arrays(tasks)
    T, fin = sgp.sgp_makespan(pd, ps, st, [3, 2, 3, 2], handoff=1.0)
    assert T == 9.0 and fin == [3.0, 6.0, 6.0, 9.0]
    assert sgp.sgp_makespan(pd, ps, st, [3, 2, 3, 2])[0] == 8.0
    with pytest.raises(sgp.SgpError):             # a predecessor after its successor
        sgp.sgp_makespan([1, -1], [-1, -1], [0, 1], [1.0, 1.0])
