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
