"""Host-side checks that need no GPU: the library loads, exports every entry point
that include/sgp.h declares, and its host-only functions behave."""
import ctypes
import os
import re

import pytest

from intra_spatial_pipelining_gb300 import build, sgp
from oracle import schedule as S

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return sgp.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "sgp.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(sgp_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported_and_bound(lib):
    names = _declared()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(sgp.ABI_FUNCTIONS) == names


def test_status_strings(lib):
    assert sgp.sgp_status_string(0) == "ok"
    for c in range(-7, 0):
        assert sgp.sgp_status_string(c) != "unknown status"


def test_struct_layouts_match_the_header(lib, tmp_path):
    """Every field offset and struct size of the ctypes mirrors equals what a C
    compiler computes from include/sgp.h."""
    import subprocess
    structs = [sgp.sgp_dims, sgp.sgp_layer, sgp.sgp_layer_dump, sgp.sgp_device_info,
               sgp.sgp_pipeline_opts]
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "sgp.h"', "int main(void){"]
    for st in structs:
        n = st.__name__
        lines.append(f'printf("{n} %zu\\n", sizeof({n}));')
        for f, _ in st._fields_:
            lines.append(f'printf("{n}.{f} %zu\\n", offsetof({n}, {f}));')
    lines.append("return 0;}")
    src = tmp_path / "abi.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "abi"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    out = dict(l.split() for l in subprocess.run([str(exe)], capture_output=True, text=True,
                                                  check=True).stdout.splitlines())
    for st in structs:
        n = st.__name__
        assert int(out[n]) == ctypes.sizeof(st), n
        for f, _ in st._fields_:
            assert int(out[f"{n}.{f}"]) == getattr(st, f).offset, f"{n}.{f}"


def test_workspace_bytes_validates(lib):
    d = sgp.make_dims(__import__("intra_spatial_pipelining_gb300.synth", fromlist=["x"]).SHAPE_GPTOSS)
    assert sgp.sgp_workspace_bytes(d, 64, 8192) > 0
    d.head_dim = 128
    assert sgp.sgp_workspace_bytes(d, 64, 8192) == 0


def test_split_enumerator_matches_the_model(lib):
    for n_sm, q, pmin in ((152, 8, 16), (148, 2, 2), (132, 8, 16), (64, 4, 4)):
        got = sgp.sgp_enumerate_splits(n_sm, q, pmin)
        ref = [p[0] for p in S.allocations(n_sm, 2, q, pmin)] if n_sm % q == 0 else None
        if ref is not None:
            assert got == ref
        assert all(pmin <= p <= n_sm - pmin and p % q == 0 for p in got)
    # the page's 148-SM, 2-SM-quantum grid has 73 two-stage allocations
    assert len(sgp.sgp_enumerate_splits(148, 2, 2)) == S.count_allocations_closed(148, 2, 2)


def _gptoss_dims():
    from intra_spatial_pipelining_gb300 import synth
    return sgp.make_dims(synth.SHAPE_GPTOSS)


def test_pipeline_create_rejects_bad_arguments_before_any_device_work(lib):
    """sgp_pipeline_create validates its arguments first: every bad argument returns
    SGP_ERR_INVALID_ARG, leaves *out NULL and records a message (no CUDA call is made)."""
    d = _gptoss_dims()
    split = (ctypes.c_int * 2)(40, 112)
    opts = sgp.make_opts()

    def create(dims, n_stages=2, micro=32, max_tokens=64, max_kv=8192, out=True):
        h = ctypes.c_void_p(12345)
        r = lib.sgp_pipeline_create(dims, split, n_stages, micro, max_tokens, max_kv,
                                    ctypes.byref(opts), ctypes.byref(h) if out else None)
        return r, h.value

    bad_dims = _gptoss_dims()
    bad_dims.head_dim = 128
    cases = [
        dict(dims=ctypes.byref(bad_dims)),                       # head_dim != 64
        dict(dims=None),                                          # dims NULL
        dict(dims=ctypes.byref(d), n_stages=0),
        dict(dims=ctypes.byref(d), n_stages=4),
        dict(dims=ctypes.byref(d), micro=24),                     # does not divide 64
        dict(dims=ctypes.byref(d), micro=0),
        dict(dims=ctypes.byref(d), micro=512, max_tokens=1024),   # more than 512 sequences
        dict(dims=ctypes.byref(d), max_kv=0),
    ]
    for c in cases:
        r, h = create(**c)
        assert r == sgp.SGP_ERR_INVALID_ARG, c
        assert h is None, c                                       # *out was reset to NULL
        assert lib.sgp_last_error().decode()
    r, _ = create(ctypes.byref(d), out=False)
    assert r == sgp.SGP_ERR_INVALID_ARG


def test_dims_checks_cover_every_documented_limit(lib):
    """check_dims, reached through sgp_workspace_bytes (0 = rejected)."""
    good = _gptoss_dims()
    assert lib.sgp_workspace_bytes(ctypes.byref(good), 64, 8192) > 0
    edits = [("hidden", 2880 + 32), ("hidden", 4096 + 64), ("inter", 100), ("n_kv_heads", 0),
             ("n_q_heads", 60), ("n_q_heads", 8 * 17), ("top_k", 0), ("top_k", 9),
             ("n_experts", 2), ("n_experts", 2048), ("n_local_experts", 0),
             ("n_local_experts", 129), ("slot_map", 2), ("path", 3), ("rope_theta", -1.0),
             ("rms_eps", 0.0), ("comm_floor_us", -1.0), ("comm_floor_us", 2e5),
             ("comm_gbps", -1.0)]
    for field, value in edits:
        d = _gptoss_dims()
        setattr(d, field, value)
        assert lib.sgp_workspace_bytes(ctypes.byref(d), 64, 8192) == 0, (field, value)
    assert lib.sgp_workspace_bytes(ctypes.byref(good), 0, 8192) == 0
    assert lib.sgp_workspace_bytes(ctypes.byref(good), 64, 0) == 0


def test_layer_calls_reject_bad_arguments_before_any_device_work(lib):
    """sgp_layer_op / sgp_layer_temporal: op index, token count, NULL pointers and alignment
    are checked before the library touches the device."""
    d = _gptoss_dims()
    layer = sgp.sgp_layer()
    buf = ctypes.create_string_buffer(4096 + 256)
    base = (ctypes.addressof(buf) + 255) & ~255
    ok_ptr = ctypes.c_void_p(base)
    odd_ptr = ctypes.c_void_p(base + 8)
    E = sgp.SGP_ERR_INVALID_ARG
    op = lambda o, T, kv, x, y, ws: lib.sgp_layer_op(ctypes.byref(d), ctypes.byref(layer), o,
                                                       kv, x, y, T, ws, 1 << 30, None)
    assert op(-1, 64, ok_ptr, ok_ptr, ok_ptr, ok_ptr) == E
    assert op(9, 64, ok_ptr, ok_ptr, ok_ptr, ok_ptr) == E
    assert op(0, 0, ok_ptr, ok_ptr, ok_ptr, ok_ptr) == E
    assert op(0, 513, ok_ptr, ok_ptr, ok_ptr, ok_ptr) == E
    assert op(0, 64, None, ok_ptr, ok_ptr, ok_ptr) == E
    assert op(0, 64, ok_ptr, None, ok_ptr, ok_ptr) == E
    assert op(0, 64, ok_ptr, ok_ptr, ok_ptr, None) == E
    assert op(0, 64, ok_ptr, odd_ptr, ok_ptr, ok_ptr) == E       # x not 16-byte aligned
    assert op(0, 64, ok_ptr, ok_ptr, ok_ptr, odd_ptr) == E       # workspace not 256-byte aligned
    # a layer with NULL weights is refused by the layer check
    assert op(0, 64, ok_ptr, ok_ptr, ok_ptr, ok_ptr) == E
    tmp = lambda T, layer_ptr, kv: lib.sgp_layer_temporal(
        ctypes.byref(d), layer_ptr, kv, ok_ptr, ok_ptr, T, None, None, ok_ptr, 1 << 30,
        None, None)
    assert tmp(64, None, ok_ptr) == E                            # no layers
    assert tmp(64, ctypes.byref(layer), None) == E               # kv_len NULL
    assert tmp(0, ctypes.byref(layer), ok_ptr) == E
    assert tmp(64, ctypes.byref(layer), ok_ptr) == E             # NULL weights


def test_pipeline_calls_on_a_null_handle(lib):
    E = sgp.SGP_ERR_INVALID_ARG
    n = ctypes.c_int(-1)
    assert lib.sgp_pipeline_sync(None) == E
    assert lib.sgp_pipeline_tasks(None, ctypes.byref(n), None, 0) == E
    assert lib.sgp_pipeline_trace(None, None, 0, ctypes.byref(n)) == E
    assert lib.sgp_pipeline_run(None, None, 1, None, None, None, 64, None, None, None) == E
    lib.sgp_pipeline_destroy(None)  # no-op


def test_noalloc_router_refuses_bad_arguments_before_any_device_work(lib):
    """The allocation-free router checks pointers, dims (hidden above 4096 included: its
    rows would not fit in shared memory) and the fixed scratch size before any CUDA call."""
    d = _gptoss_dims()
    buf = ctypes.create_string_buffer(4096 + 256)
    base = (ctypes.addressof(buf) + 255) & ~255
    ok, odd = ctypes.c_void_p(base), ctypes.c_void_p(base + 8)
    E = sgp.SGP_ERR_INVALID_ARG

    def call(dims, T=64, h=ok, u=ok, idx=ok, w=ok):
        return lib.sgp_router_topk_noalloc(ctypes.byref(dims), h, ok, ok, None, T, u, idx, w,
                                           None)
    assert call(d, h=None) == E
    assert call(d, idx=None) == E
    assert call(d, h=odd) == E
    assert call(d, u=odd) == E
    assert call(d, T=0) == E
    big = _gptoss_dims()
    big.hidden = 4096 + 64
    assert call(big) == E
    wide = _gptoss_dims()
    wide.n_experts = 1024
    assert call(wide, T=257) == E                 # 257 x 1024 logits exceed the scratch
