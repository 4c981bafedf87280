"""Host-side logic of bench.py (no GPU): the peak a kernel is held against and the
algorithmic bytes of a step, which enter the reported roofline."""
import numpy as np

import bench
from block_sparse_masked_02_gb300 import workloads as W

PEAKS = {"hbm_gbs": 6769.1, "bf16_tflops": 1879.0, "bf16_tflops_sustained": 1706.1, "source": "measured"}


def test_peak_is_burst_without_power_cap():
    peak, src = bench.select_peak(PEAKS, {"sm_mhz": 2070.0, "reasons": []})
    assert peak == 1879.0 and "burst" in src


def test_peak_is_sustained_under_power_cap():
    peak, src = bench.select_peak(PEAKS, {"sm_mhz": 1500.0, "reasons": ["sw_power_cap"]})
    assert peak == 1706.1 and "sw_power_cap" in src


def _causal_map(nt, full_diag=False):
    bm = np.zeros((1, 1, nt, nt), dtype=np.int8)
    for qt in range(nt):
        bm[0, 0, qt, :qt + 1] = 1
    return bm


def test_algorithmic_bytes_dense_topk():
    wl = W.scaled(W.WORKLOADS["n16384_hq16_hkv4"], B=1, Nq=1024, Nk=1024, Hq=4, Hkv=1)
    bm = _causal_map(8)
    b = bench.algorithmic_bytes(wl, bm)
    tiles = 36  # causally allowed (and here all active) tiles of an 8 x 8 map
    assert b["mask"] == tiles * 128 * 128 * 2
    assert b["bias"] == 2 * tiles * 128 * 128 * 2
    assert b["dbias"] == 1024 * 1024 * 2
    io = 2 * (4 * 1024 * 4 * 128 + 4 * 1024 * 1 * 128) + 4 * 4 * 1024
    assert b["io"] == io
    assert b["total"] == b["mask"] + b["bias"] + b["dbias"] + io


def test_algorithmic_bytes_column_ranges_no_bias():
    wl = W.scaled(W.WORKLOADS["docmask_b2_n32768"], Nq=1024, Nk=1024)
    bm = _causal_map(8)
    b = bench.algorithmic_bytes(wl, bm)
    assert b["mask"] == wl.B * wl.Hkv * 1024 * 2 * 4  # two int32 per key column
    assert b["bias"] == 0 and b["dbias"] == 0
