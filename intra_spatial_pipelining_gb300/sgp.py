"""Thin ctypes binding of libsgp.so: argument marshalling only.

Every function here has the name of the C entry point it forwards to (see
``include/sgp.h``).  Tensors are passed as device pointers (``tensor.data_ptr()``)
and streams as ``torch.cuda.Stream.cuda_stream``.  There is no fallback: when the
library is missing, loading raises.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libsgp.so")

SGP_OK = 0
SGP_ERR_INVALID_ARG = -1
SGP_ERR_UNSUPPORTED = -2
SGP_ERR_CUDA = -3
SGP_ERR_TIMEOUT = -4
SGP_ERR_OOM = -5
SGP_ERR_HANDOFF = -6
SGP_ERR_DEVICE_BOUNDS = -7

OPS = ("rmsnorm_attn", "qkv", "attention", "oproj", "router", "dispatch", "expert_up",
       "expert_down", "combine")
N_OPS = len(OPS)
PATH_AUTO, PATH_GEMV, PATH_TC = 0, 1, 2


class sgp_dims(C.Structure):
    _fields_ = [("hidden", C.c_int), ("n_q_heads", C.c_int), ("n_kv_heads", C.c_int),
                ("head_dim", C.c_int), ("n_experts", C.c_int), ("top_k", C.c_int),
                ("n_local_experts", C.c_int), ("inter", C.c_int), ("rms_eps", C.c_float),
                ("slot_map", C.c_int), ("path", C.c_int), ("gemv_max_tokens", C.c_int),
                ("rope_theta", C.c_float), ("comm_floor_us", C.c_float), ("comm_gbps", C.c_float)]


class sgp_layer(C.Structure):
    _fields_ = [("g_attn", C.c_void_p), ("w_qkv", C.c_void_p), ("w_o", C.c_void_p),
                ("g_mlp", C.c_void_p), ("w_router", C.c_void_p), ("router_bias", C.c_void_p),
                ("w_gate_up", C.c_void_p), ("w_down", C.c_void_p), ("k_cache", C.c_void_p),
                ("v_cache", C.c_void_p), ("kv_cap", C.c_int), ("window", C.c_int)]


class sgp_layer_dump(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("a", "q", "o", "h", "u", "logits", "slot_offsets",
                                          "pair_pos", "z", "y")]


class sgp_device_info(C.Structure):
    _fields_ = [("sm_count", C.c_int), ("cc_major", C.c_int), ("cc_minor", C.c_int),
                ("green_ctx_supported", C.c_int), ("sm_min_partition", C.c_int),
                ("sm_alignment", C.c_int), ("l2_bytes", C.c_size_t)]


class sgp_pipeline_opts(C.Structure):
    _fields_ = [("custom_cut", C.c_int), ("stage_of_op", (C.c_int * N_OPS) * 2),
                ("use_green_contexts", C.c_int), ("green_ctx_flags", C.c_int),
                ("serpentine_experts", C.c_int), ("wait_timeout_ns", C.c_uint64),
                ("fault_inject", C.c_uint32), ("fault_task", C.c_int),
                ("programmatic_launch", C.c_int), ("trace", C.c_int),
                ("weight_reuse", C.c_int), ("l2_prefetch_mb", C.c_int),
                ("stage_lanes", C.c_int), ("stage_times_shared", C.c_int)]


_lib = None

_SIGS = {
    "sgp_device_info_get": (C.c_int, [C.POINTER(sgp_device_info)]),
    "sgp_status_string": (C.c_char_p, [C.c_int]),
    "sgp_last_error": (C.c_char_p, []),
    "sgp_workspace_bytes": (C.c_size_t, [C.POINTER(sgp_dims), C.c_int, C.c_int]),
    "sgp_layer_temporal": (C.c_int, [C.POINTER(sgp_dims), C.POINTER(sgp_layer), C.c_void_p,
                                     C.c_void_p, C.c_void_p, C.c_int, C.c_void_p, C.c_void_p,
                                     C.c_void_p, C.c_size_t, C.POINTER(sgp_layer_dump),
                                     C.c_void_p]),
    "sgp_stack_temporal": (C.c_int, [C.POINTER(sgp_dims), C.POINTER(sgp_layer), C.c_int,
                                     C.c_void_p, C.c_void_p, C.c_void_p, C.c_int, C.c_void_p,
                                     C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p]),
    "sgp_layer_op": (C.c_int, [C.POINTER(sgp_dims), C.POINTER(sgp_layer), C.c_int, C.c_void_p,
                               C.c_void_p, C.c_void_p, C.c_int, C.c_void_p, C.c_size_t,
                               C.c_void_p]),
    "sgp_status_from_workspace": (C.c_int, [C.c_void_p, C.c_void_p]),
    "sgp_router_topk_noalloc": (C.c_int, [C.POINTER(sgp_dims), C.c_void_p, C.c_void_p,
                                          C.c_void_p, C.c_void_p, C.c_int, C.c_void_p,
                                          C.c_void_p, C.c_void_p, C.c_void_p]),
    "sgp_pipeline_create": (C.c_int, [C.POINTER(sgp_dims), C.POINTER(C.c_int), C.c_int, C.c_int,
                                      C.c_int, C.c_int, C.POINTER(sgp_pipeline_opts),
                                      C.POINTER(C.c_void_p)]),
    "sgp_pipeline_run": (C.c_int, [C.c_void_p, C.POINTER(sgp_layer), C.c_int, C.c_void_p,
                                   C.c_void_p, C.c_void_p, C.c_int, C.c_void_p, C.c_void_p,
                                   C.c_void_p]),
    "sgp_pipeline_sync": (C.c_int, [C.c_void_p]),
    "sgp_pipeline_stage_times": (C.c_int, [C.c_void_p, C.POINTER(sgp_layer), C.c_int, C.c_void_p,
                                           C.c_void_p, C.c_void_p, C.c_int, C.c_int,
                                           C.POINTER(C.c_float)]),
    "sgp_pipeline_tasks": (C.c_int, [C.c_void_p, C.POINTER(C.c_int), C.POINTER(C.c_int32),
                                     C.c_int]),
    "sgp_pipeline_trace": (C.c_int, [C.c_void_p, C.POINTER(C.c_uint64), C.c_int,
                                     C.POINTER(C.c_int)]),
    "sgp_pipeline_trace_sms": (C.c_int, [C.c_void_p, C.POINTER(C.c_uint32), C.c_int,
                                         C.POINTER(C.c_int)]),
    "sgp_pipeline_task_spans": (C.c_int, [C.c_void_p, C.POINTER(C.c_uint64), C.c_int,
                                          C.POINTER(C.c_int)]),
    "sgp_pipeline_destroy": (None, [C.c_void_p]),
    "sgp_enumerate_splits": (C.c_int, [C.c_int, C.c_int, C.c_int, C.POINTER(C.c_int), C.c_int]),
    "sgp_pipeline_balance": (C.c_int, [C.POINTER(sgp_dims), C.POINTER(sgp_layer), C.c_int,
                                       C.c_void_p, C.c_void_p, C.c_void_p, C.c_int, C.c_int,
                                       C.c_int, C.c_int, C.c_int, C.POINTER(sgp_pipeline_opts),
                                       C.POINTER(C.c_int), C.POINTER(C.c_int),
                                       C.POINTER(C.c_float), C.c_int, C.POINTER(C.c_int)]),
}

_SIGS["sgp_makespan"] = (C.c_int, [C.c_int, C.POINTER(C.c_int32), C.POINTER(C.c_int32),
                                   C.POINTER(C.c_int32), C.POINTER(C.c_double), C.c_double,
                                   C.POINTER(C.c_double), C.POINTER(C.c_double)])
_SIGS["sgp_pipeline_predict"] = (C.c_int, [C.c_void_p, C.POINTER(sgp_layer), C.c_int, C.c_void_p,
                                           C.c_void_p, C.c_void_p, C.c_int, C.c_float,
                                           C.POINTER(C.c_float), C.POINTER(C.c_float)])
_SIGS["sgp_pipeline_refine"] = (C.c_int, [C.POINTER(sgp_dims), C.POINTER(sgp_layer), C.c_int,
                                          C.c_void_p, C.c_void_p, C.c_void_p, C.c_int, C.c_int,
                                          C.c_int, C.c_int, C.c_int, C.c_int, C.c_int,
                                          C.POINTER(sgp_pipeline_opts), C.POINTER(C.c_int),
                                          C.POINTER(C.c_float), C.POINTER(C.c_int)])
ALLOC_OBJECTIVE = C.CFUNCTYPE(C.c_double, C.POINTER(C.c_int), C.c_int, C.c_void_p)
_SIGS["sgp_refine_allocation"] = (C.c_int, [C.c_int, C.POINTER(C.c_int), C.c_int, C.c_int,
                                            C.c_int, ALLOC_OBJECTIVE, C.c_void_p,
                                            C.POINTER(C.c_double)])

ABI_FUNCTIONS = tuple(_SIGS)


def lib() -> C.CDLL:
    """The loaded library (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libsgp.so not built ({LIB_PATH}); run "
                               "`python -m intra_spatial_pipelining_gb300.build`")
        h = C.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(h, name)
            f.restype = res
            f.argtypes = args
        _lib = h
    return _lib


class SgpError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = lib().sgp_status_string(code).decode()
        detail = lib().sgp_last_error().decode()
        super().__init__(f"{where}: {msg} ({code}) {detail}")


def check(code: int, where: str) -> int:
    if code != SGP_OK:
        raise SgpError(code, where)
    return code


def _p(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


# --------------------------------------------------------------------------------------
# structure builders
# --------------------------------------------------------------------------------------
def make_dims(shape, path: int = PATH_AUTO, gemv_max_tokens: int = 2,
              comm_floor_us: float = 0.0, comm_gbps: float = 0.0) -> sgp_dims:
    """Layer dimensions.  comm_floor_us / comm_gbps > 0 turn on the virtual communication
    kernels (3 us and 900 GB/s are the pages' model of a B200 NVLink deployment).  The
    default path threshold sends only single-sequence batches to the GEMV path, which is
    where it beats the tcgen05 GEMM in temporal execution (measured over 36 layers)."""
    return sgp_dims(shape.hidden, shape.n_q_heads, shape.n_kv_heads, shape.head_dim,
                    shape.n_experts, shape.top_k, shape.n_local_experts, shape.inter,
                    shape.rms_eps, 0 if shape.slot_map == "mod" else 1, path, gemv_max_tokens,
                    float(getattr(shape, "rope_theta", 0.0)), float(comm_floor_us),
                    float(comm_gbps))


def make_layer(w: dict, k_cache, v_cache, window: int) -> sgp_layer:
    return sgp_layer(_p(w["g_attn"]), _p(w["w_qkv"]), _p(w["w_o"]), _p(w["g_mlp"]),
                     _p(w["w_router"]), _p(w.get("router_bias")), _p(w["w_gate_up"]),
                     _p(w["w_down"]), _p(k_cache), _p(v_cache), int(k_cache.shape[2]),
                     int(window))


def layer_array(layers: Sequence[sgp_layer]):
    arr = (sgp_layer * len(layers))()
    for i, l in enumerate(layers):
        arr[i] = l
    return arr


def make_opts(stage_of_op=None, use_green_contexts: int = 0, green_ctx_flags: int = 0,
              serpentine_experts: int = 0, wait_timeout_ns: int = 0, fault_inject: int = 0,
              fault_task: int = 0, programmatic_launch: int = 0,
              trace: int = 0, weight_reuse: int = 0, l2_prefetch_mb: int = 0,
              stage_lanes: int = 0, stage_times_shared: int = 0) -> sgp_pipeline_opts:
    o = sgp_pipeline_opts()
    if stage_of_op is not None:
        o.custom_cut = 1
        for s in range(2):
            for op in range(N_OPS):
                o.stage_of_op[s][op] = int(stage_of_op[s][op])
    o.use_green_contexts = use_green_contexts
    o.green_ctx_flags = green_ctx_flags
    o.serpentine_experts = serpentine_experts
    o.wait_timeout_ns = wait_timeout_ns
    o.fault_inject = fault_inject
    o.fault_task = fault_task
    o.programmatic_launch = programmatic_launch
    o.trace = trace
    o.weight_reuse = weight_reuse
    o.l2_prefetch_mb = l2_prefetch_mb
    o.stage_lanes = stage_lanes
    o.stage_times_shared = stage_times_shared
    return o


# --------------------------------------------------------------------------------------
# entry points (same names as the C ABI)
# --------------------------------------------------------------------------------------
def sgp_device_info_get() -> sgp_device_info:
    info = sgp_device_info()
    check(lib().sgp_device_info_get(C.byref(info)), "sgp_device_info_get")
    return info


def sgp_status_string(code: int) -> str:
    return lib().sgp_status_string(code).decode()


def sgp_workspace_bytes(dims: sgp_dims, n_tokens: int, max_kv_len: int) -> int:
    return int(lib().sgp_workspace_bytes(C.byref(dims), n_tokens, max_kv_len))


def sgp_layer_temporal(dims, layer: sgp_layer, kv_len, x_in, x_out, n_tokens: int, topk_idx,
                       topk_w, workspace, dump: Optional[sgp_layer_dump] = None,
                       stream=None) -> int:
    return check(lib().sgp_layer_temporal(
        C.byref(dims), C.byref(layer), _p(kv_len), _p(x_in), _p(x_out), n_tokens, _p(topk_idx),
        _p(topk_w), _p(workspace), workspace.numel() * workspace.element_size(),
        C.byref(dump) if dump is not None else None, _stream(stream)), "sgp_layer_temporal")


def sgp_stack_temporal(dims, layers, kv_len, x_in, x_out, n_tokens: int, topk_idx, topk_w,
                       workspace, stream=None) -> int:
    arr = layer_array(layers)
    return check(lib().sgp_stack_temporal(
        C.byref(dims), arr, len(layers), _p(kv_len), _p(x_in), _p(x_out), n_tokens,
        _p(topk_idx), _p(topk_w), _p(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)), "sgp_stack_temporal")


def sgp_layer_op(dims, layer: sgp_layer, op: int, kv_len, x_in, x_out, n_tokens: int,
                 workspace, stream=None) -> int:
    return check(lib().sgp_layer_op(C.byref(dims), C.byref(layer), op, _p(kv_len), _p(x_in),
                                    _p(x_out), n_tokens, _p(workspace),
                                    workspace.numel() * workspace.element_size(),
                                    _stream(stream)), "sgp_layer_op")


def sgp_router_topk_noalloc(dims, h, g_mlp, w_router, router_bias, n_tokens: int, u_out,
                            topk_idx, topk_w, stream=None) -> int:
    return check(lib().sgp_router_topk_noalloc(C.byref(dims), _p(h), _p(g_mlp), _p(w_router),
                                               _p(router_bias), n_tokens, _p(u_out),
                                               _p(topk_idx), _p(topk_w), _stream(stream)),
                 "sgp_router_topk_noalloc")


def sgp_status_from_workspace(workspace, stream=None) -> int:
    return lib().sgp_status_from_workspace(_p(workspace), _stream(stream))


def sgp_pipeline_create(dims, sm_split: Sequence[int], n_stages: int, microbatch: int,
                        max_tokens: int, max_kv_len: int,
                        opts: Optional[sgp_pipeline_opts] = None) -> int:
    split = (C.c_int * max(1, len(sm_split)))(*sm_split)
    h = C.c_void_p()
    check(lib().sgp_pipeline_create(C.byref(dims), split, n_stages, microbatch, max_tokens,
                                    max_kv_len, C.byref(opts) if opts is not None else None,
                                    C.byref(h)), "sgp_pipeline_create")
    return h.value


def sgp_pipeline_run(p, layers, kv_len, x_in, x_out, n_tokens: int, topk_idx=None, topk_w=None,
                     stream=None) -> int:
    arr = layers if isinstance(layers, C.Array) else layer_array(layers)
    return check(lib().sgp_pipeline_run(p, arr, len(arr), _p(kv_len), _p(x_in), _p(x_out),
                                        n_tokens, _p(topk_idx), _p(topk_w), _stream(stream)),
                 "sgp_pipeline_run")


def sgp_pipeline_sync(p) -> int:
    return lib().sgp_pipeline_sync(p)


def sgp_pipeline_stage_times(p, layers, kv_len, x_in, x_out, n_tokens: int, n_stages: int,
                             reps: int = 5) -> list:
    arr = layers if isinstance(layers, C.Array) else layer_array(layers)
    t = (C.c_float * n_stages)()
    check(lib().sgp_pipeline_stage_times(p, arr, len(arr), _p(kv_len), _p(x_in), _p(x_out),
                                         n_tokens, reps, t), "sgp_pipeline_stage_times")
    return list(t)


def sgp_pipeline_tasks(p) -> list:
    n = C.c_int()
    check(lib().sgp_pipeline_tasks(p, C.byref(n), None, 0), "sgp_pipeline_tasks")
    rows = (C.c_int32 * (5 * max(1, n.value)))()
    check(lib().sgp_pipeline_tasks(p, C.byref(n), rows, n.value), "sgp_pipeline_tasks")
    return [tuple(rows[5 * i:5 * i + 5]) for i in range(n.value)]


def sgp_pipeline_trace(p):
    """Launch trace of the last run as an int64 array [n_pairs][2] of (start_ns, end_ns),
    indexed [layer][microbatch][op][part] (flattened); zeros mark launches that do not exist."""
    import numpy as np
    n = C.c_int()
    check(lib().sgp_pipeline_trace(p, None, 0, C.byref(n)), "sgp_pipeline_trace")
    out = np.zeros((max(1, n.value), 2), dtype=np.uint64)
    check(lib().sgp_pipeline_trace(p, out.ctypes.data_as(C.POINTER(C.c_uint64)), n.value,
                                   C.byref(n)), "sgp_pipeline_trace")
    return out[:n.value].astype(np.int64)


def sgp_pipeline_trace_sms(p):
    """SM masks of the last run's launches as a uint32 array [n_entries][8] (bit %smid set
    for every SM a CTA of that launch ran on), indexed like sgp_pipeline_trace."""
    import numpy as np
    n = C.c_int()
    check(lib().sgp_pipeline_trace_sms(p, None, 0, C.byref(n)), "sgp_pipeline_trace_sms")
    out = np.zeros((max(1, n.value), 8), dtype=np.uint32)
    check(lib().sgp_pipeline_trace_sms(p, out.ctypes.data_as(C.POINTER(C.c_uint32)), n.value,
                                       C.byref(n)), "sgp_pipeline_trace_sms")
    return out[:n.value]


def sgp_pipeline_task_spans(p):
    """Measured (start_ns, end_ns) of every task of the last run, in task order, as an int64
    array [n_tasks][2]."""
    import numpy as np
    n = C.c_int()
    check(lib().sgp_pipeline_task_spans(p, None, 0, C.byref(n)), "sgp_pipeline_task_spans")
    out = np.zeros((max(1, n.value), 2), dtype=np.uint64)
    check(lib().sgp_pipeline_task_spans(p, out.ctypes.data_as(C.POINTER(C.c_uint64)), n.value,
                                        C.byref(n)), "sgp_pipeline_task_spans")
    return out[:n.value].astype(np.int64)


def handoff_gaps_us(p):
    """Cross-stage handoff latencies of the last run (traced pipeline): for every task whose
    data predecessor ran on another stage and finished after the task's stage predecessor
    (so the handoff was what the task waited for), its start minus that data predecessor's
    end, in us."""
    import numpy as np
    spans = sgp_pipeline_task_spans(p)
    tasks = sgp_pipeline_tasks(p)
    gaps = []
    for i, (st, _, _, pd, ps) in enumerate(tasks):
        if pd < 0 or tasks[pd][0] == st:
            continue
        if ps >= 0 and spans[ps, 1] > spans[pd, 1]:
            continue
        gaps.append((spans[i, 0] - spans[pd, 1]) * 1e-3)
    return np.array(gaps, dtype=np.float64)


def sgp_refine_allocation(p0: Sequence[int], quantum: int, p_min: int, objective,
                          pass_limit: int = 0):
    """Pairwise-line refinement of the allocation p0 under objective(p: tuple) -> float
    (lower is better; negative = cannot evaluate).  Returns (allocation, value, evaluations)."""
    n = len(p0)
    p = (C.c_int * n)(*p0)
    err = []

    def _f(pp, nn, _ctx):
        try:
            return float(objective(tuple(pp[i] for i in range(nn))))
        except Exception as e:          # an exception must not unwind through C
            err.append(e)
            return -1.0
    cb = ALLOC_OBJECTIVE(_f)
    t = C.c_double()
    r = lib().sgp_refine_allocation(n, p, quantum, p_min, pass_limit, cb, None, C.byref(t))
    if err:
        raise err[0]
    if r < 0:
        raise SgpError(r, "sgp_refine_allocation")
    return tuple(p), t.value, r


def sgp_makespan(pred_data, pred_stage, stage, tau, handoff: float = 0.0):
    """Eq. 4-5 on a task DAG (lists in a topological order, -1 = no predecessor); returns
    (makespan, per-task finish times)."""
    n = len(tau)
    arr = lambda v, t: (t * max(1, n))(*v)
    fin = (C.c_double * max(1, n))()
    T = C.c_double()
    check(lib().sgp_makespan(n, arr(pred_data, C.c_int32), arr(pred_stage, C.c_int32),
                             arr(stage, C.c_int32), arr(tau, C.c_double), float(handoff),
                             C.byref(T), fin), "sgp_makespan")
    return T.value, list(fin[:n])


def sgp_pipeline_predict(p, layers, kv_len, x_in, x_out, n_tokens: int, n_stages: int,
                         handoff_us: float = 0.0):
    """Eq. 4-5 makespan (us) predicted from task durations measured under contention, and
    each stage's summed task durations."""
    arr = layers if isinstance(layers, C.Array) else layer_array(layers)
    t = C.c_float()
    st = (C.c_float * n_stages)()
    check(lib().sgp_pipeline_predict(p, arr, len(arr), _p(kv_len), _p(x_in), _p(x_out), n_tokens,
                                     float(handoff_us), C.byref(t), st), "sgp_pipeline_predict")
    return t.value, list(st)


def sgp_pipeline_refine(dims, layers, kv_len, x_in, x_out, n_tokens: int, split: Sequence[int],
                        microbatch: int, max_kv_len: int, quantum: int = 8, reps: int = 3,
                        pass_limit: int = 0, opts: Optional[sgp_pipeline_opts] = None):
    """Measured pairwise-line refinement of `split`; returns (split, us, evaluations)."""
    arr = layers if isinstance(layers, C.Array) else layer_array(layers)
    n = len(split)
    sp = (C.c_int * n)(*split)
    t = C.c_float()
    ev = C.c_int()
    check(lib().sgp_pipeline_refine(C.byref(dims), arr, len(arr), _p(kv_len), _p(x_in),
                                    _p(x_out), n_tokens, n, microbatch, max_kv_len, quantum, reps,
                                    pass_limit, C.byref(opts) if opts is not None else None, sp,
                                    C.byref(t), C.byref(ev)), "sgp_pipeline_refine")
    return list(sp), t.value, ev.value


def sgp_pipeline_destroy(p) -> None:
    if p:
        lib().sgp_pipeline_destroy(p)


def sgp_enumerate_splits(n_sm: int, quantum: int, p_min: int) -> list:
    n = lib().sgp_enumerate_splits(n_sm, quantum, p_min, None, 0)
    if n < 0:
        raise SgpError(n, "sgp_enumerate_splits")
    out = (C.c_int * max(1, n))()
    lib().sgp_enumerate_splits(n_sm, quantum, p_min, out, n)
    return list(out[:n])


def sgp_pipeline_balance(dims, layers, kv_len, x_in, x_out, n_tokens: int, microbatch: int,
                         max_kv_len: int, quantum: int = 8, reps: int = 3,
                         opts: Optional[sgp_pipeline_opts] = None, max_out: int = 64):
    arr = layers if isinstance(layers, C.Array) else layer_array(layers)
    best = C.c_int()
    splits = (C.c_int * max_out)()
    t = (C.c_float * (2 * max_out))()
    n = C.c_int()
    check(lib().sgp_pipeline_balance(C.byref(dims), arr, len(arr), _p(kv_len), _p(x_in),
                                     _p(x_out), n_tokens, microbatch, max_kv_len, quantum, reps,
                                     C.byref(opts) if opts is not None else None, C.byref(best),
                                     splits, t, max_out, C.byref(n)), "sgp_pipeline_balance")
    k = min(n.value, max_out)
    return best.value, [(splits[i], t[2 * i], t[2 * i + 1]) for i in range(k)]
