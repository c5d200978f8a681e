"""Host-side arithmetic of the measurement scripts: the algorithmic byte count of an
iteration (the roofline numerator of every DRAM percentage) written out by hand for the
36-layer slice, and the same count in bench.py and in the profiler-range script."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from intra_spatial_pipelining_gb300 import pipebench, synth  # noqa: E402


def test_c2_bytes_written_out_by_hand():
    """36 layers x (W_qkv 5120 x 2880 + W_o 2880 x 4096 + W_r 128 x 2880 + 4 experts x 3 x
    2880 x 2880 + two gains), bf16; 18 full layers read 64 x 8 KV heads x 8192 positions x
    64 x (K, V) bf16, 18 sliding layers the last 128 positions; every layer appends one K and
    one V row per sequence and head.  Activations are the small rest (about 1 %: 9.2 MB per
    layer, the token rows in and out of each op and the routed rows)."""
    wl = synth.WORKLOADS["gptoss_36l"]
    weights = 36 * 2 * (5120 * 2880 + 2880 * 4096 + 128 * 2880 + 4 * 3 * 2880 * 2880 + 2 * 2880)
    kv_full = 18 * 64 * 8 * 8192 * 64 * 2 * 2
    kv_slide = 18 * 64 * 8 * 128 * 64 * 2 * 2
    append = 36 * 64 * 8 * 64 * 2 * 2
    total = bench.algorithmic_bytes(wl)
    rest = total - (weights + kv_full + kv_slide + append)
    assert weights == 9_104_348_160          # 9.10 GB
    assert kv_full == 19_327_352_832         # 19.33 GB
    assert 0 < rest < 0.02 * total
    # the 4.28 ms floor at the measured 6,795.1 GB/s
    assert abs(total / 6795.1e9 * 1e3 - 4.28) < 0.005


def test_bench_and_range_script_count_alike():
    for wl in (synth.WORKLOADS["gptoss_36l"].with_(n_layers=2), synth.WORKLOADS["paper_32k"],
               synth.sweep_workload(16, n_layers=3)):
        lens = synth.kv_len(wl, 0, "cpu").tolist()
        assert bench.algorithmic_bytes(wl, lens) == pipebench.algorithmic_bytes(wl, lens)
