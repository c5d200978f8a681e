"""Schedule model of the spatial pipeline: the augmented task DAG and its makespan.

TEST INFRASTRUCTURE ONLY (see ``oracle/layer.py``): used by the tests to check
the product's task graph and its measured task timestamps.

Follows "SubGPU Pipelining: Intra-GPU Fine-Grained Spatial Parallelism for LLM
Inference":
  * Section 3.1, Eq. 1: segment-to-stage binding rho_w(k) (w = 1: the last
    segment shares stage 1).
  * Section 3.2: a task i = (layer, microbatch, segment) runs on stage
    rho_w(segment); its data predecessors are the task of the previous segment
    (or of the last segment of the previous layer) for the same microbatch; its
    stage predecessor is the task before it on the same stage in a fixed global
    dispatch order that is a topological order of the data edges.
  * Eq. 4-5: A_i = max(max_{j in data(i)} C_j, max_{j in stage(i)} C_j),
    C_i = A_i + tau_i, makespan T = max_i C_i (an empty maximum is zero).
  * Section 4.2, Eq. 7 and the illustrative counts that follow it: the number
    of cut-and-binding choices of an operator chain and of SM allocations in
    quanta.
  * Section 4.2, Algorithm 2: pairwise-line SM-allocation refinement (the best
    one-quantum transfer between two stages, then a doubling/halving line search
    along that donor-receiver pair, repeated until no transfer improves).
"""
from __future__ import annotations

import itertools
from math import comb


def binding(k: int, n_segments: int, w: int) -> int:
    """rho_w(k) for 1-based segment k of K = n_segments segments (Eq. 1)."""
    return 1 if (w == 1 and k == n_segments) else k


def build_tasks(n_layers: int, n_micro: int, n_segments: int, w: int = 0, lanes: int = 1):
    """Tasks of the unrolled forward pass in the global dispatch order
    (layer-major, then microbatch, then segment).

    lanes = 1 is the pages' model: one FIFO per stage.  lanes = 2 gives each stage one FIFO
    per microbatch parity (two streams sharing the stage's SM pool, as the pages' prototype
    runs two stream rows per green context, Section 5.3); the stage edge of a task then
    points to the previous task of its own lane.

    Returns a list of dicts with keys: id, layer, micro, seg (1-based), stage,
    data (list of predecessor ids), stage_pred (id or None)."""
    order = []
    for l in range(n_layers):
        for mu in range(n_micro):
            for k in range(1, n_segments + 1):
                order.append((l, mu, k))
    index = {key: i for i, key in enumerate(order)}
    last_on_stage = {}
    tasks = []
    for i, (l, mu, k) in enumerate(order):
        if k > 1:
            data = [index[(l, mu, k - 1)]]
        elif l > 0:
            data = [index[(l - 1, mu, n_segments)]]
        else:
            data = []
        st = binding(k, n_segments, w)
        lane = (st, mu % lanes)
        tasks.append({"id": i, "layer": l, "micro": mu, "seg": k, "stage": st,
                      "data": data, "stage_pred": last_on_stage.get(lane)})
        last_on_stage[lane] = i
    return tasks


def makespan(tasks, tau) -> tuple[float, list, list]:
    """Eq. 4-5 over tasks in a topological order.  tau[i] is task i's duration.
    Returns (T, A, C)."""
    A = [0.0] * len(tasks)
    C = [0.0] * len(tasks)
    for t in tasks:
        i = t["id"]
        preds = list(t["data"])
        if t["stage_pred"] is not None:
            preds.append(t["stage_pred"])
        A[i] = max((C[j] for j in preds), default=0.0)
        C[i] = A[i] + tau[i]
    return (max(C) if C else 0.0), A, C


def longest_path(tasks, tau) -> float:
    """The same makespan computed independently as the longest weighted path of
    the augmented DAG (memoised recursion over predecessors)."""
    memo = {}

    def finish(i):
        if i not in memo:
            t = tasks[i]
            preds = list(t["data"]) + ([t["stage_pred"]] if t["stage_pred"] is not None else [])
            memo[i] = tau[i] + max((finish(j) for j in preds), default=0.0)
        return memo[i]

    return max((finish(i) for i in range(len(tasks))), default=0.0)


def steady_state_period(stage_times) -> float:
    """Per-microbatch period of a full pipeline in steady state: the slowest stage."""
    return max(stage_times)


# ---------------------------------------------------------------------------
# counting (Section 4.2)
# ---------------------------------------------------------------------------
def chain_cuts(n_ops: int, n_segments: int):
    """All ways to cut a chain of n_ops operators into n_segments non-empty
    contiguous segments; each cut is a tuple of segment lengths."""
    for bars in itertools.combinations(range(1, n_ops), n_segments - 1):
        edges = (0,) + bars + (n_ops,)
        yield tuple(edges[i + 1] - edges[i] for i in range(n_segments))


def count_cut_bindings(n_ops: int, n_stages: int) -> int:
    """|C_D(G)| + |C_{D+1}(G)| for a chain G (one-to-one and boundary-reuse
    bindings), counted by enumeration."""
    return sum(1 for _ in chain_cuts(n_ops, n_stages)) + \
        sum(1 for _ in chain_cuts(n_ops, n_stages + 1))


def allocations(n_sm: int, n_stages: int, quantum: int, p_min: int = 0):
    """Ordered SM allocations p (sum = n_sm, each a positive multiple of quantum
    and >= p_min), by enumeration."""
    if n_sm % quantum:
        return
    q = n_sm // quantum
    for bars in itertools.combinations(range(1, q), n_stages - 1):
        edges = (0,) + bars + (q,)
        p = tuple((edges[i + 1] - edges[i]) * quantum for i in range(n_stages))
        if min(p) >= max(p_min, quantum):
            yield p


def count_allocations(n_sm: int, n_stages: int, quantum: int) -> int:
    return sum(1 for _ in allocations(n_sm, n_stages, quantum))


def count_allocations_closed(n_sm: int, n_stages: int, quantum: int) -> int:
    """Stars and bars: compositions of n_sm/quantum into n_stages positive parts."""
    return comb(n_sm // quantum - 1, n_stages - 1)


# ---------------------------------------------------------------------------
# Section 4.2, Algorithm 2: pairwise-line SM-allocation refinement
# ---------------------------------------------------------------------------
def transfer(p, d: int, r: int, z: int, g: int):
    """p^{d->r}[z]: z*g SMs move from donor stage d to receiver stage r."""
    q = list(p)
    q[d] -= z * g
    q[r] += z * g
    return tuple(q)


def pairwise_line(f, feasible, p, g: int, passes=None):
    """Algorithm 2 in the pages' steps.  f(p) is the objective (lower is better),
    feasible(p) the membership test of P, p the initial allocation, g the SM quantum and
    passes the pass limit L (None = until no improving move).  Returns the refined
    allocation and its objective value."""
    p = tuple(p)
    t = f(p)
    n = len(p)
    k = 0
    while passes is None or k < passes:
        k += 1
        M = [(d, r) for d in range(n) for r in range(n) if d != r and feasible(transfer(p, d, r, 1, g))]
        if not M:
            return p, t
        d, r = min(M, key=lambda dr: f(transfer(p, dr[0], dr[1], 1, g)))
        z, h = 1, 1
        t_line = f(transfer(p, d, r, 1, g))
        if t_line >= t:
            return p, t
        while h > 0:
            z2 = z + h
            q = transfer(p, d, r, z2, g)
            if feasible(q) and f(q) < t_line:
                z, t_line, h = z2, f(q), 2 * h
            else:
                h //= 2
        p, t = transfer(p, d, r, z, g), t_line
    return p, t
