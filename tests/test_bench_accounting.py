"""The benchmark's work accounting, on the CPU: the algorithmic K/V, Q and output bytes
(the numerator of the roofline's achieved bandwidth) and the attention FLOPs, checked by
brute-force counts of what each query row must read and multiply, and against the
per-workload figures of the measurement plan (K/V bytes 2 * Hkv * d * bytes per element
* sum_b (T_b + 1 + D_b); FLOPs 4 * d per (query row, visible key))."""
import os
import sys

import numpy as np
import pytest

from speculative_decoding_verification_gqa_gb300 import synth

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def _brute(w, T, D, window=0):
    """Positions read per (sequence, KV head): the union of every window row's visible
    keys; multiply-adds: every (query head, window row, visible key)."""
    elem = 1 if w.kv_dtype == "fp8_e4m3" else 2
    positions, pairs = 0, 0
    for Tb, Db in zip(T.tolist(), D.tolist()):
        seen = set()
        for i in range(Db + 1):
            lo = 0 if window == 0 else max(0, Tb + i - window + 1)
            keys = range(lo, Tb + i + 1)
            seen.update(keys)
            pairs += len(keys)
        positions += len(seen)
    kv = 2 * w.Hkv * w.d * elem * positions
    qo = 2 * int(np.sum(D + 1)) * w.Hq * w.d * 2
    return kv, qo, 4 * w.Hq * w.d * pairs


@pytest.mark.parametrize("window", [0, 1, 5, 64, 1000])
@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
def test_bytes_and_flops_match_a_brute_force_count(window, kv):
    w = synth.Workload("a", B=5, Hq=8, Hkv=2, d=64, D=0, T=0, V=8, p=0.5, kv_dtype=kv)
    T = np.array([0, 1, 37, 300, 999], dtype=np.int32)
    D = np.array([0, 3, 7, 1, 15], dtype=np.int32)
    kv_b, qo_b, fl = _brute(w, T, D, window)
    assert bench.algorithmic_bytes(w, T, D, window=window) == (kv_b, qo_b)
    if window == 0:
        assert bench.flops(w, T, D) == fl


def test_measured_workloads_figures():
    """c2: 16 x (8192 + 32) positions x 8 heads x 128 x 2 bytes x (K, V) = 538,968,064 B;
    c3: the same count at one byte per element = 537,133,056 B; c4: 1.074 GB at every draft
    length swept. FLOPs count every visible key of every row (prefix plus the window's
    triangle), within 0.3% of the 4 B Hq W T d approximation (68.7 G on c2, 137.4 G on
    c3)."""
    for cfg, kv_want, gf_approx in (("c2", 538_968_064, 68.72), ("c3", 537_133_056, 137.44)):
        w = synth.CONFIGS[cfg]
        T, D, _ = synth.lengths(w, 0)
        kv_b, qo_b = bench.algorithmic_bytes(w, T, D)
        assert kv_b == kv_want
        assert qo_b == 2 * int(np.sum(D + 1)) * w.Hq * w.d * 2
        Wn, Tn = int(D[0]) + 1, int(T[0])
        exact = 4 * w.Hq * w.d * w.B * (Wn * Tn + Wn * (Wn + 1) // 2)
        assert bench.flops(w, T, D) == exact
        approx = 4 * w.B * w.Hq * Wn * Tn * w.d
        assert abs(approx / 1e9 - gf_approx) < 0.01
        assert 0 < exact / approx - 1 < 0.003
    w = synth.CONFIGS["c4"]
    for Dc in synth.C4_SWEEP_D:
        T, D, _ = synth.lengths(w, 0, D=Dc)
        kv_b, _ = bench.algorithmic_bytes(w, T, D)
        assert abs(kv_b / 1e9 - 1.074) < 0.005


def test_window_bytes_on_the_side_figure():
    """The 4096-position window on c2: the last window row sees T + 31 - 4095 .. T + 31, the
    first T - 4095 .. T, so every sequence needs positions T - 4095 .. T + 31 (4127 of
    them): 270,467,072 bytes of K/V, the side figure's kv_bytes."""
    w = synth.CONFIGS["c2"]
    T, D, _ = synth.lengths(w, 0)
    kv_b, _ = bench.algorithmic_bytes(w, T, D, window=4096)
    assert kv_b == 2 * 8 * 128 * 2 * 16 * 4127 == 270_467_072
