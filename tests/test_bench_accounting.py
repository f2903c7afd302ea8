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


def test_roofline_bound_is_the_slower_of_hbm_and_tensor_time():
    """The bound is whichever of (bytes / HBM peak) and (FLOPs / tensor peak of their types)
    is larger, and frac = that time / the kernel's time. c2 (bf16, G(1+D) = 128): HBM, 80.8
    us of bytes against 35.3 us of FLOPs at 6780 GB/s and 1948 TFLOP/s. A contraction of 64
    rows per key at d = 128 over 1 GB is tensor-bound."""
    w = synth.CONFIGS["c2"]
    T, D, _ = synth.lengths(w, 0)
    kv_b, qo_b = bench.algorithmic_bytes(w, T, D)
    fl = bench.flops(w, T, D)
    r = bench.roofline_record(kv_b, qo_b, fl, 100e-6, 6780.0, 1948.2, "bf16", "tcgen05")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == 6780.0
    assert abs(r["t_hbm_us"] - (kv_b + qo_b) / 6780e9 * 1e6) < 0.01
    assert abs(r["t_tensor_us"] - fl / 1948.2e12 * 1e6) < 0.01
    assert abs(r["frac"] - r["t_hbm_us"] / 100.0) < 1e-4
    assert abs(r["achieved"] - (kv_b + qo_b) / 100e-6 / 1e9) < 0.1
    # tensor-bound: FLOPs far above the bytes' worth
    r = bench.roofline_record(1e9, 0, 4e15, 3e-3, 6780.0, 1948.2, "bf16", "tcgen05")
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert abs(r["peak"] - 1948.2) < 0.1 and abs(r["achieved"] - 4e15 / 3e-3 / 1e12) < 0.1
    assert abs(r["frac"] - (4e15 / 1948.2e12) / 3e-3) < 1e-4


def test_fp8_tensor_time_uses_the_e4m3_rate_for_qk_only():
    """FP8 K/V on the tcgen05 kernel: Q K^T (half the FLOPs) at twice the bf16 rate, P V
    (the other half) at the bf16 rate; 0.75 of the bf16 time. The mma.sync kernel decodes
    to f16: the full bf16 time. c3 stays HBM-bound (79.8 us of bytes vs 52.9 us)."""
    fl = 1e12
    t16 = bench.tensor_seconds(fl, "bf16", "tcgen05", 1000.0)
    assert abs(t16 - 1e-3) < 1e-12
    assert abs(bench.tensor_seconds(fl, "fp8_e4m3", "tcgen05", 1000.0) - 0.75e-3) < 1e-12
    assert abs(bench.tensor_seconds(fl, "fp8_e4m3", "mma.sync", 1000.0) - 1e-3) < 1e-12
    w = synth.CONFIGS["c3"]
    T, D, _ = synth.lengths(w, 0)
    kv_b, qo_b = bench.algorithmic_bytes(w, T, D)
    r = bench.roofline_record(kv_b, qo_b, bench.flops(w, T, D), 120e-6, 6780.0, 1948.2,
                              "fp8_e4m3", "tcgen05")
    assert r["bound"] == "hbm" and 52 < r["t_tensor_us"] < 54 and 79 < r["t_hbm_us"] < 81


def test_ncu_traffic_is_dropped_when_the_sources_change(monkeypatch):
    h = bench.kernel_source_hash()
    assert len(h) == 16 and h == bench.kernel_source_hash()
    monkeypatch.setitem(bench.NCU_TRAFFIC, ("c2", None, "tcgen05"), (h, 12345))
    monkeypatch.setitem(bench.NCU_TRAFFIC, ("c3", None, "tcgen05"), ("0" * 16, 999))
    assert bench.ncu_traffic("c2", None, "tcgen05") == 12345
    assert bench.ncu_traffic("c3", None, "tcgen05") is None      # another kernel version
    assert bench.ncu_traffic("c4", 7, "tcgen05") is None         # never captured


def test_source_hash_ignores_comments_but_not_code():
    """The capture key of the attention kernel's ncu traffic names the code, not its
    comments: comment and layout edits keep it, any change to code or to a literal (inline
    PTX lives in strings) does not."""
    src = 'int a = 1; // note\n/* block */ asm("ld.global // x");\n'
    assert bench.code_text(src) == bench.code_text('int a = 1;\n   asm("ld.global // x");')
    assert bench.code_text(src) != bench.code_text('int a = 2; asm("ld.global // x");')
    assert bench.code_text(src) != bench.code_text('int a = 1; asm("ld.global // y");')
    assert bench.code_text("char c = '\"'; // q\nx;") == "char c = '\"'; x;"
