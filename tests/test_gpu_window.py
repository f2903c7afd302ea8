"""GPU parity of sliding-window verify attention (spec_verify_attn with sliding_window =
W): window row i sees keys max(0, T+i-W+1) .. T+i. Small ragged shapes against the full
oracle for windows below, across and beyond tile boundaries; row tiles of one sequence
with different first tiles; cache rows before the window holding NaN; the workloads at
full size with a 4096-position window on sampled units."""
import numpy as np
import pytest

import speculative_decoding_verification_gqa_gb300 as sv
from speculative_decoding_verification_gqa_gb300 import synth

from gpu_util import assert_close, bf16_to_f64, ensure_built, gpu_attn, oracle_attn

pytestmark = pytest.mark.gpu


@pytest.fixture(params=[1, 2], ids=["mma", "tcgen05"])
def kernel(request):
    ensure_built()
    lib = sv.api.load_library()
    prev = lib.sv_set_attn_kernel(request.param)
    if prev < 0:
        pytest.skip("kernel not built")
    yield request.param
    lib.sv_set_attn_kernel(prev)


def _small(B, Hq, Hkv, d, T, D, kv="bf16", seed=0):
    w = synth.Workload("sw", B=B, Hq=Hq, Hkv=Hkv, d=d, D=0, T=0, V=8, p=0.5, kv_dtype=kv,
                       outlier_prob=0.001 if kv != "bf16" else 0.0)
    return w, synth.attn_inputs(w, seed, seq_lens=np.array(T), draft_len=np.array(D))


RAGGED = dict(B=4, Hq=8, Hkv=2, d=128, T=(1000, 37, 300, 5000), D=(5, 0, 15, 9))


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
@pytest.mark.parametrize("W", [1, 2, 7, 64, 127, 128, 129, 300, 1001, 4096, 6000])
def test_ragged_batch_against_full_oracle(kernel, kv, W):
    w, x = _small(kv=kv, seed=W, **RAGGED)
    assert_close(gpu_attn(x, window=W), oracle_attn(w, x, window=W))


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
@pytest.mark.parametrize("W", [5, 40, 200])
def test_row_tiles_with_different_first_tiles(kernel, kv, W):
    """G * (1 + D) = 256 query rows per KV head: two row tiles whose smallest window rows
    (0 and 16) start their windows in different key tiles."""
    w, x = _small(B=2, Hq=32, Hkv=4, d=128, T=(500, 130), D=(31, 31), kv=kv, seed=3)
    assert_close(gpu_attn(x, window=W), oracle_attn(w, x, window=W))


@pytest.mark.parametrize("d", [64, 128])
def test_head_dim_64_and_short_prefixes(kernel, d):
    w, x = _small(B=3, Hq=16, Hkv=2, d=d, T=(0, 3, 513), D=(4, 2, 1), seed=5)
    for W in (1, 3, 6, 100):
        assert_close(gpu_attn(x, window=W), oracle_attn(w, x, window=W))


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
def test_rows_before_the_window_may_hold_nan(kernel, kv):
    """Cache rows of positions before T - W + 1 are never used: NaN there (K and V) must
    not reach the output, including the rows that share a key tile with the window."""
    w, x = _small(B=3, Hq=8, Hkv=2, d=128, T=(700, 260, 90), D=(7, 3, 0), kv=kv, seed=9)
    W = 150
    ref = oracle_attn(w, x, window=W)
    k, v = x["k"].copy(), x["v"].copy()
    nan = 0x7F if kv == "fp8_e4m3" else 0x7FC0  # E4M3 NaN code / bf16 quiet NaN
    ko = 0
    for T, D in zip(x["seq_lens"].tolist(), x["draft_len"].tolist()):
        if T - W + 1 > 0:
            k[ko:ko + T - W + 1] = nan
            v[ko:ko + T - W + 1] = nan
        ko += T + D + 1
    got = gpu_attn(dict(x, k=k, v=v), window=W)
    assert np.isfinite(bf16_to_f64(got)).all()
    assert_close(got, ref)


def test_window_covering_every_key_equals_no_window(kernel):
    """W >= T + D + 1 for every sequence: the same tiles as without a window, so the same
    bits."""
    w, x = _small(**RAGGED, seed=11)
    full = gpu_attn(x)
    assert np.array_equal(gpu_attn(x, window=5016), full)
    assert np.array_equal(gpu_attn(x, window=1 << 30), full)


def test_window_of_one_returns_the_rows_own_value(kernel):
    w, x = _small(B=2, Hq=8, Hkv=2, d=128, T=(333, 0), D=(6, 2), seed=12)
    got = bf16_to_f64(gpu_attn(x, window=1))
    v = bf16_to_f64(x["v"])
    qo = ko = 0
    for T, D in zip(x["seq_lens"].tolist(), x["draft_len"].tolist()):
        for i in range(D + 1):
            for h in range(w.Hq):
                assert np.array_equal(got[qo + i, h], v[ko + T + i, h // w.G])
        qo += D + 1
        ko += T + D + 1


_cache = {}


def _full(cfg):
    if cfg not in _cache:
        _cache.clear()
        w = synth.CONFIGS[cfg]
        _cache[cfg] = (w, synth.attn_inputs(w, 1))
    return _cache[cfg]


@pytest.mark.parametrize("cfg", ["c2", "c3", "c5"])
def test_full_size_4096_window_sampled_units(kernel, cfg):
    """The workloads' shapes with Mistral 7B's 4096-position window, on sampled
    (sequence, KV head) units."""
    w, x = _full(cfg)
    W = 4096
    got = gpu_attn(x, window=W)
    rng = np.random.default_rng(17)
    B = len(x["seq_lens"])
    units = sorted({(0, 0), (B - 1, w.Hkv - 1), (int(np.argmin(x["seq_lens"])), 0)} |
                   {(int(rng.integers(B)), int(rng.integers(w.Hkv))) for _ in range(3)})
    assert_close(got, oracle_attn(w, x, units=units, window=W))
    assert np.isfinite(bf16_to_f64(got)).all()
