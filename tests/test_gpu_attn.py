"""GPU parity of spec_verify_attn against the fp64 oracle (max-abs <= 1e-2, normwise
max-rel <= 2e-2): small shapes computed in full (several tiles, ragged tails, edge cases),
the five workloads at full size on sampled (sequence, KV head) units, and device-side
checks."""
import zlib

import numpy as np
import pytest
import torch

import speculative_decoding_verification_gqa_gb300 as sv
from speculative_decoding_verification_gqa_gb300 import synth

from gpu_util import (assert_close, bf16_to_f64, dev_attn, ensure_built, gpu_attn,
                      oracle_attn)

pytestmark = pytest.mark.gpu


def _kernels():
    ensure_built()
    ks = [1]
    prev = sv.api.load_library().sv_set_attn_kernel(2)
    if prev >= 0:
        sv.api.load_library().sv_set_attn_kernel(prev)
        ks.append(2)
    return ks


@pytest.fixture(params=[1, 2], ids=["mma", "tcgen05"])
def kernel(request):
    if request.param not in _kernels():
        pytest.skip("kernel not built")
    prev = sv.set_attn_kernel(request.param)
    yield request.param
    sv.set_attn_kernel(prev)


def _small(B, Hq, Hkv, d, T, D, kv="bf16", seed=0):
    w = synth.Workload("s", B=B, Hq=Hq, Hkv=Hkv, d=d, D=0, T=0, V=8, p=0.5, kv_dtype=kv,
                       outlier_prob=0.001 if kv != "bf16" else 0.0)
    return w, synth.attn_inputs(w, seed, seq_lens=np.array(T), draft_len=np.array(D))


SMALL = {
    "c1": dict(B=1, Hq=4, Hkv=1, d=64, T=(256,), D=(3,)),
    "ragged": dict(B=3, Hq=8, Hkv=2, d=128, T=(1000, 37, 129), D=(5, 0, 15)),
    "decode_D0": dict(B=2, Hq=32, Hkv=8, d=128, T=(300, 777), D=(0, 0)),
    "G1_mha": dict(B=2, Hq=4, Hkv=4, d=128, T=(200, 64), D=(3, 7)),
    "empty_prefix": dict(B=2, Hq=8, Hkv=2, d=64, T=(0, 1), D=(4, 0)),
    "tile_edges": dict(B=4, Hq=8, Hkv=2, d=128, T=(63, 64, 127, 128), D=(0, 1, 0, 1)),
    "rows_136": dict(B=2, Hq=32, Hkv=4, d=128, T=(500, 260), D=(16, 16)),
    "rows_192": dict(B=2, Hq=32, Hkv=4, d=128, T=(700, 129), D=(23, 23)),
    "rows_256": dict(B=1, Hq=32, Hkv=4, d=128, T=(400,), D=(31,)),
    "llama3_8b_shape": dict(B=2, Hq=32, Hkv=8, d=128, T=(1500, 333), D=(31, 31)),
    "d64_ragged": dict(B=3, Hq=16, Hkv=2, d=64, T=(513, 5, 2049), D=(8, 2, 1)),
    # ~7 tiles per CTA on 152 CTAs: every ring stage and buffer parity is reused
    "tiles_per_cta": dict(B=2, Hq=16, Hkv=2, d=128, T=(40000, 30000), D=(7, 3)),
}


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
@pytest.mark.parametrize("name", list(SMALL))
def test_small_shapes_full_oracle(kernel, name, kv):
    w, x = _small(kv=kv, seed=zlib.crc32(name.encode()) % 1000, **SMALL[name])
    got = gpu_attn(x)
    ref = oracle_attn(w, x)
    assert_close(got, ref)


@pytest.mark.parametrize("window", [0, 300])
@pytest.mark.parametrize("name", ["c1", "ragged", "tile_edges", "rows_136", "rows_256",
                                  "llama3_8b_shape", "d64_ragged", "tiles_per_cta"])
def test_kv_ring_modes_bit_identical(name, window):
    """bf16 K/V on the tcgen05 kernel with paired K + V stages and with separate K and V
    rings (by default chosen by the call's shape): the same output bits either way, and
    the oracle's values; with and without a sliding window (whose V rows before the window
    are cleared in the ring's stage)."""
    if 2 not in _kernels():
        pytest.skip("kernel not built")
    prev_k = sv.set_attn_kernel(2)
    try:
        w, x = _small(kv="bf16", seed=zlib.crc32(name.encode()) % 1000 + 7, **SMALL[name])
        outs = []
        for mode in (0, 1):
            prev = sv.api.set_kv_rings(mode)
            try:
                outs.append(gpu_attn(x, window=window))
            finally:
                sv.api.set_kv_rings(prev)
        assert np.array_equal(outs[0], outs[1])
        assert_close(outs[1], oracle_attn(w, x, window=window))
    finally:
        sv.set_attn_kernel(prev_k)


def test_rows_beyond_packed_batch_untouched(kernel):
    w, x = _small(B=2, Hq=8, Hkv=2, d=128, T=(100, 50), D=(3, 2))
    q, k, v, sc, T, D = dev_attn(x)
    rows = q.shape[0]
    qbig = torch.zeros((rows + 5, 8, 128), dtype=torch.bfloat16, device="cuda")
    qbig[:rows] = q
    out = torch.full_like(qbig, 7.0)
    sv.spec_verify_attn(qbig, k, v, T, D, max_draft_len=3, max_seq_len=100, out=out)
    torch.cuda.synchronize()
    assert (out[rows:] == 7.0).all()
    ref = oracle_attn(w, x)
    assert_close(out[:rows].contiguous().view(torch.int16).cpu().numpy().view(np.uint16), ref)


def test_repeatable_and_workspace_reuse(kernel):
    w, x = _small(B=3, Hq=16, Hkv=4, d=128, T=(3000, 10, 900), D=(7, 3, 0))
    q, k, v, sc, T, D = dev_attn(x)
    ws = sv.new_workspace(sv.verify_workspace_bytes(sv.api.attn_desc(q, k, 3, 7, 3000)))
    o1 = sv.spec_verify_attn(q, k, v, T, D, max_draft_len=7, max_seq_len=3000, workspace=ws)
    o2 = sv.spec_verify_attn(q, k, v, T, D, max_draft_len=7, max_seq_len=3000, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)
    assert sv.workspace_status(ws) == 0


@pytest.mark.parametrize("name", ["ragged", "d64_ragged", "empty_prefix", "c1"])
def test_stale_workspace_is_never_read(kernel, name):
    """Partials are only read where this call wrote them: a workspace full of NaN bytes
    (flag word zeroed) must give the same result as a fresh one, including ragged batches
    with fewer tiles than CTAs (some CTAs then own no tile)."""
    w, x = _small(seed=5, **SMALL[name])
    q, k, v, sc, T, D = dev_attn(x)
    md, ms = int(x["draft_len"].max()), int(x["seq_lens"].max())
    nbytes = sv.verify_workspace_bytes(sv.api.attn_desc(q, k, len(x["seq_lens"]), md, ms))
    ws = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device="cuda")
    ws[:256] = 0
    out = sv.spec_verify_attn(q, k, v, T, D, max_draft_len=md, max_seq_len=ms, workspace=ws)
    torch.cuda.synchronize()
    assert sv.workspace_status(ws) == 0
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    assert_close(got, oracle_attn(w, x))


def test_device_side_length_check(kernel):
    w, x = _small(B=2, Hq=8, Hkv=2, d=128, T=(100, 50), D=(3, 2))
    q, k, v, sc, T, D = dev_attn(x)
    ws = sv.new_workspace(sv.verify_workspace_bytes(sv.api.attn_desc(q, k, 2, 2, 100)))
    out = torch.full_like(q, 3.0)
    sv.spec_verify_attn(q, k, v, T, D, max_draft_len=2, max_seq_len=100, out=out,
                        workspace=ws)                     # D_0 = 3 > max_draft_len = 2
    assert sv.workspace_status(ws, clear=True) == 8
    assert (out == 3.0).all()
    out2 = sv.spec_verify_attn(q, k, v, T, D, max_draft_len=3, max_seq_len=99, out=out,
                               workspace=ws)              # T_0 = 100 > max_seq_len = 99
    assert sv.workspace_status(ws, clear=True) == 8
    assert (out2 == 3.0).all()
    small_q = q[:5].contiguous()                         # q_rows 5 < sum W = 7
    with pytest.raises(ValueError):
        sv.spec_verify_attn(small_q, k, v, T, D, max_draft_len=3, max_seq_len=100,
                            out=torch.empty_like(q))      # out shape != q shape
    sv.spec_verify_attn(small_q, k, v, T, D, max_draft_len=3, max_seq_len=100, workspace=ws)
    assert sv.workspace_status(ws, clear=True) == 8


# ------------------------------------------------------------------ full-size workloads

_cache = {}


def _full(cfg, D=None):
    key = (cfg, D)
    if key not in _cache:
        _cache.clear()
        w = synth.CONFIGS[cfg]
        if D is None:
            x = synth.attn_inputs(w, 1)
        else:
            T, Dv, _ = synth.lengths(w, 1, D=D)
            x = synth.attn_inputs(w, 1, seq_lens=T, draft_len=Dv)
        _cache[key] = (w, x)
    return _cache[key]


def _sample_units(w, x, n, seed):
    rng = np.random.default_rng(seed)
    B = len(x["seq_lens"])
    picks = {(0, 0), (B - 1, w.Hkv - 1)}
    if w.ragged:  # include the longest and the shortest sequence
        picks.add((int(np.argmax(x["seq_lens"])), 0))
        picks.add((int(np.argmin(x["seq_lens"])), w.Hkv - 1))
    while len(picks) < n:
        picks.add((int(rng.integers(B)), int(rng.integers(w.Hkv))))
    return sorted(picks)


@pytest.mark.parametrize("cfg,D", [("c1", None), ("c2", None), ("c3", None)]
                         + [("c4", Dc) for Dc in synth.C4_SWEEP_D] + [("c5", None)])
def test_full_size_sampled_units(kernel, cfg, D):
    w, x = _full(cfg, D)
    got = gpu_attn(x)
    units = None if cfg == "c1" else _sample_units(w, x, 6, seed=7)
    ref = oracle_attn(w, x, units=units)
    ma, mr = assert_close(got, ref)
    # every packed row was written with finite values
    assert np.isfinite(bf16_to_f64(got)).all()


# ------------------------------------------------------------------ closed forms on the GPU

def _bits(x):
    return synth.bf16_bits(np.asarray(x, dtype=np.float32))


def _run_raw(q, k, v, T, D):
    x = dict(q=q, k=k, v=v, kv_scale=None, seq_lens=np.asarray(T, dtype=np.int32),
             draft_len=np.asarray(D, dtype=np.int32))
    return bf16_to_f64(gpu_attn(x))


@pytest.mark.parametrize("T,D", [(300, 9), (250, 15), (127, 1), (0, 31)])
def test_window_mask_with_dominant_window_keys(kernel, T, D):
    """Window keys score far above the prefix, so row i averages the V rows of the window
    keys it may see, positions T..T+i. V column 0 holds the window index j, so row i must
    return i/2 exactly; a mask off by one key moves it by 0.5."""
    Hq, Hkv, d = 8, 2, 128
    W = D + 1
    q = np.zeros((W, Hq, d), dtype=np.float32)
    q[:, :, 0] = 4.0
    k = np.zeros((T + W, Hkv, d), dtype=np.float32)
    k[T:, :, 0] = 64.0                           # score 4*64/sqrt(128) = 22.6 vs 0
    vals = np.zeros((T + W, Hkv, d), dtype=np.float32)
    vals[T:, :, 0] = np.arange(W)[:, None]
    vals[T:, :, 1] = 1.0
    out = _run_raw(_bits(q), _bits(k), _bits(vals), [T], [D])
    for i in range(W):
        assert np.abs(out[i, :, 0] - i / 2.0).max() <= 0.05, (i, out[i, :, 0])
        assert np.abs(out[i, :, 1] - 1.0).max() <= 1e-2


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
def test_running_max_grows_on_some_rows_only(kernel, kv):
    """Scores of half the query heads jump by ~12 (log2 units) from one 128-key tile to
    the next while the other half stay flat, so the online-softmax rescale of O happens on
    some rows of a warp and not on others, tile after tile."""
    Hq, Hkv, d, T, D = 8, 2, 128, 700, 7
    W = D + 1
    rng = np.random.default_rng(3)
    q = rng.standard_normal((W, Hq, d)).astype(np.float32) * 0.25
    q[:, 0::2, 0] = 8.0                                # even heads see the ramp
    q[:, 1::2, 0] = 0.0
    k = rng.standard_normal((T + W, Hkv, d)).astype(np.float32) * 0.25
    k[:, :, 0] = (np.arange(T + W) // 128)[:, None] * 12.0
    v = rng.standard_normal((T + W, Hkv, d)).astype(np.float32)
    w = synth.Workload("r", B=1, Hq=Hq, Hkv=Hkv, d=d, D=0, T=0, V=8, p=0.5, kv_dtype=kv)
    x = dict(q=_bits(q))
    x.update(dict(k=_bits(k), v=_bits(v), kv_scale=None) if kv == "bf16" else _fp8_kv(k, v))
    x.update(seq_lens=np.array([T], dtype=np.int32), draft_len=np.array([D], dtype=np.int32))
    assert_close(gpu_attn(x), oracle_attn(w, x))


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
def test_row_maximum_at_every_position_of_a_half_tile(kernel, kv):
    """Query row r (of 128: 16 window positions x 8 heads) meets one dominant key per
    128-key tile, at key r of the tile, so across the rows the maximum of a warpgroup's
    64-key half sits at each of its 64 positions: a score left out of the maximum would
    leave 2^32 in P (an overflow in the 16-bit P) instead of 1."""
    Hq, Hkv, d, T, D = 8, 1, 128, 256, 15
    W = D + 1
    rng = np.random.default_rng(17)
    q = np.zeros((W, Hq, d), dtype=np.float32)
    for i in range(W):
        for h in range(Hq):
            q[i, h, i * Hq + h] = 16.0                 # row r = i*G + h: channel r
    k = np.zeros((T + W, Hkv, d), dtype=np.float32)
    for key in range(T):
        k[key, 0, key % 128] = 16.0                    # keys r and r + 128 match row r
    v = rng.standard_normal((T + W, Hkv, d)).astype(np.float32)
    w = synth.Workload("m", B=1, Hq=Hq, Hkv=Hkv, d=d, D=0, T=0, V=8, p=0.5, kv_dtype=kv)
    x = dict(q=_bits(q))
    x.update(dict(k=_bits(k), v=_bits(v), kv_scale=None) if kv == "bf16" else _fp8_kv(k, v))
    x.update(seq_lens=np.array([T], dtype=np.int32), draft_len=np.array([D], dtype=np.int32))
    got = gpu_attn(x)
    assert np.isfinite(bf16_to_f64(got)).all()
    assert_close(got, oracle_attn(w, x))


def _fp8_kv(k, v):
    """Per-KV-head E4M3 quantisation of float K and V (scale = absmax / 448)."""
    sk = np.abs(k).max(axis=(0, 2)) / 448.0
    sv_ = np.abs(v).max(axis=(0, 2)) / 448.0
    return dict(k=synth.e4m3_codes(k / sk[None, :, None]),
                v=synth.e4m3_codes(v / sv_[None, :, None]),
                kv_scale=np.stack([sk, sv_]).astype(np.float32))


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
def test_query_rows_of_wide_dynamic_range(kernel, kv):
    """Query rows scaled by 2^-12 .. 2^8, the elements of each row spread over 2^-10 .. 2^2:
    the large rows give sharp score distributions, in which an error of 1/16 in a Q element
    moves P by tens of percent, and the tiny rows average V almost uniformly. On the 8-bit
    score path this checks the per-row power-of-two scale and both E4M3 terms of Q."""
    Hq, Hkv, d, T, D = 8, 1, 128, 400, 3
    W = D + 1
    rng = np.random.default_rng(11)
    q = rng.standard_normal((W, Hq, d)) * np.exp2(rng.uniform(-10, 2, (W, Hq, d)))
    q *= np.exp2(np.array([-12, -4, 0, 1, 2, 3, 6, 8], dtype=np.float64))[None, :, None]
    k = rng.standard_normal((T + W, Hkv, d)).astype(np.float32)
    v = rng.standard_normal((T + W, Hkv, d)).astype(np.float32)
    w = synth.Workload("q", B=1, Hq=Hq, Hkv=Hkv, d=d, D=0, T=0, V=8, p=0.5, kv_dtype=kv)
    x = dict(q=_bits(q), seq_lens=np.array([T], dtype=np.int32),
             draft_len=np.array([D], dtype=np.int32))
    x.update(dict(k=_bits(k), v=_bits(v), kv_scale=None) if kv == "bf16" else _fp8_kv(k, v))
    assert_close(gpu_attn(x), oracle_attn(w, x))


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
def test_nan_rows_after_the_last_sequence(kernel, kv):
    """K/V tensors longer than the packed batch, the extra rows full of NaN codes: the last
    sequence's last tile overlaps them, and they must not reach its output (P is 0 there,
    but 0 x NaN is NaN)."""
    w, x = _small(B=2, Hq=8, Hkv=2, d=128, T=(300, 190), D=(5, 3), kv=kv, seed=4)
    pad = 200
    for name in ("k", "v"):
        a = x[name]
        fill = 0x7F if a.dtype == np.uint8 else 0x7FC0  # E4M3 NaN / bf16 quiet NaN
        x[name] = np.concatenate([a, np.full((pad,) + a.shape[1:], fill, dtype=a.dtype)])
    got = gpu_attn(x)
    assert np.isfinite(bf16_to_f64(got)).all()
    assert_close(got, oracle_attn(w, x))


def test_constant_values_select_the_kv_group(kernel):
    """V constant per KV head -> query head h returns the constant of KV head h // G."""
    B, Hq, Hkv, d, T, D = 3, 32, 4, 128, 500, 7
    rng = np.random.default_rng(1)
    n_kv = B * (T + D + 1)
    q = _bits(rng.standard_normal((B * (D + 1), Hq, d)))
    k = _bits(rng.standard_normal((n_kv, Hkv, d)))
    c = np.array([1.0, -2.0, 3.5, 0.25], dtype=np.float32)
    v = _bits(np.broadcast_to(c[None, :, None], (n_kv, Hkv, d)))
    out = _run_raw(q, k, v, [T] * B, [D] * B)
    expect = np.repeat(c, Hq // Hkv)[None, :, None]
    assert np.abs(out - expect).max() <= 1e-2


def test_dominant_key_wins(kernel):
    """One key scoring far above the others returns its V row, for a key in the prefix and
    for the last window key (which only the last window row may see)."""
    Hq, Hkv, d, T, D = 4, 1, 64, 700, 3
    W = D + 1
    q = np.zeros((W, Hq, d), dtype=np.float32)
    q[:, :, 0] = 8.0
    k = np.zeros((T + W, Hkv, d), dtype=np.float32)
    k[333, 0, 0] = 16.0
    v = np.random.default_rng(2).standard_normal((T + W, Hkv, d)).astype(np.float32)
    vb = _bits(v)
    out = _run_raw(_bits(q), _bits(k), vb, [T], [D])
    assert np.abs(out - bf16_to_f64(vb)[333, 0][None, None, :]).max() <= 1e-2
    k2 = np.zeros_like(k)
    k2[T + D, 0, 0] = 16.0                      # visible to window row D only
    out2 = _run_raw(_bits(q), _bits(k2), vb, [T], [D])
    assert np.abs(out2[D] - bf16_to_f64(vb)[T + D, 0][None, :]).max() <= 1e-2
    assert np.abs(out2[0] - bf16_to_f64(vb)[T + D, 0][None, :]).max() > 0.1


# ------------------------------------------------------------- unit-to-CTA policies

@pytest.fixture(params=[0, 1, 2, 3, -1], ids=["split", "k1", "k2", "k3", "model"])
def unit_ctas(request):
    prev = sv.set_unit_ctas(request.param)
    yield request.param
    sv.set_unit_ctas(prev)


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
@pytest.mark.parametrize("name", ["ragged", "rows_256", "d64_ragged", "tile_edges", "c1"])
def test_every_unit_cta_policy(kernel, unit_ctas, name, kv):
    """The split tile line, k CTAs per unit (k = 1, 2, 3: equal parts, the last unit's end
    included) and the model's choice give the oracle's result."""
    w, x = _small(kv=kv, seed=21, **SMALL[name])
    assert_close(gpu_attn(x), oracle_attn(w, x))


@pytest.mark.parametrize("k", [1, 2])
def test_unit_cta_policy_on_a_full_size_workload(kernel, k):
    """c3 (64 units of 257 tiles) with 1 and 2 CTAs per unit, on sampled units."""
    prev = sv.set_unit_ctas(k)
    try:
        w, x = _full("c3")
        got = gpu_attn(x)
    finally:
        sv.set_unit_ctas(prev)
    assert_close(got, oracle_attn(w, x, units=[(0, 0), (7, 7), (3, 5)]))


# ------------------------------------------------------- many sequences (plan chunks)

@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
def test_many_short_ragged_sequences(kernel, kv):
    """700 sequences (more than the plan kernel handles in one pass over its threads):
    ragged prefixes and draft lengths, several units per CTA on the split line."""
    rng = np.random.default_rng(41)
    B = 700
    T = rng.integers(0, 400, size=B)
    D = rng.integers(0, 8, size=B)
    w, x = _small(B=B, Hq=8, Hkv=2, d=128, T=tuple(T), D=tuple(D), kv=kv, seed=41)
    got = gpu_attn(x)
    units = [(0, 0), (255, 1), (256, 0), (511, 1), (512, 0), (699, 1)] + \
            [(int(b), int(rng.integers(2))) for b in rng.integers(0, B, size=6)]
    assert_close(got, oracle_attn(w, x, units=units))
    assert np.isfinite(bf16_to_f64(got)).all()


def test_many_sequences_with_two_row_tiles(kernel):
    """300 sequences with G (1 + D) = 136 rows each: every sequence has two row tiles, so
    the plan reorders the units row-tile-major over several passes of its threads."""
    B = 300
    w, x = _small(B=B, Hq=8, Hkv=1, d=128, T=(150,) * B, D=(16,) * B, seed=43)
    got = gpu_attn(x)
    units = [(0, 0), (1, 0), (255, 0), (256, 0), (299, 0), (137, 0)]
    assert_close(got, oracle_attn(w, x, units=units))


def test_many_sequences_with_a_sliding_window(kernel):
    rng = np.random.default_rng(47)
    B = 520
    T = rng.integers(100, 700, size=B)
    D = rng.integers(0, 16, size=B)
    w, x = _small(B=B, Hq=8, Hkv=2, d=128, T=tuple(T), D=tuple(D), seed=47)
    got = gpu_attn(x, window=200)
    units = [(0, 0), (300, 1), (519, 1), (257, 0)]
    assert_close(got, oracle_attn(w, x, units=units, window=200))
