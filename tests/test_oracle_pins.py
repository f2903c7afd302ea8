"""Pins for the fp64 oracle: each check ties it to something other than itself (the
pages' printed values, closed forms, library routines for special cases, invariants of
the definitions, brute force on tiny inputs). CPU only."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_gqa_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits_of(x):
    """float values exactly representable in bf16 -> bf16 bit patterns (test helper)."""
    return synth.bf16_bits(np.asarray(x, dtype=np.float32))


def _decode_bf16(bits):
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def _small(B=2, Hq=4, Hkv=2, d=16, T=(5, 9), D=(2, 0), seed=0, kv="bf16"):
    w = synth.Workload("pin", B=B, Hq=Hq, Hkv=Hkv, d=d, D=0, T=0, V=8, p=0.5, kv_dtype=kv,
                       outlier_prob=0.001 if kv != "bf16" else 0.0)
    return w, synth.attn_inputs(w, seed, seq_lens=np.array(T), draft_len=np.array(D))


def _run(w, x, **kw):
    return oracle.verify_attn(x["q"], x["k"], x["v"], x["seq_lens"], x["draft_len"],
                              Hq=w.Hq, Hkv=w.Hkv, d=w.d, kv_scale=x["kv_scale"], **kw)


# ---------------------------------------------------------------- format decoders

def test_bf16_decoder_matches_torch():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 1 << 16, size=4000, dtype=np.uint16)
    bits = bits[((bits >> 7) & 0xFF) != 0xFF]  # drop inf / NaN patterns
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16_to_f64(int(b)) for b in bits])
    assert np.array_equal(got, ref)


def test_e4m3_decoder_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_f64(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert nan.sum() == 2  # 0x7F and 0xFF
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_e4m3_decoder_golden_points():
    with open(os.path.join(GOLDEN, "e4m3_points.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            code, val = line.split()
            got = oracle.e4m3_to_f64(int(code, 16))
            assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val))


# ---------------------------------------------------------------- attention

@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
@pytest.mark.parametrize("tile", [1, 3, 8, 64])
def test_online_softmax_equals_materialised(kv, tile):
    """The page states the online update gives the whole-table softmax exactly."""
    w, x = _small(kv=kv, T=(37, 3, 64), D=(5, 0, 7), B=3, seed=2)
    full = _run(w, x)
    onl = oracle.verify_attn_online(x["q"], x["k"], x["v"], x["seq_lens"], x["draft_len"],
                                    tile=tile, Hq=w.Hq, Hkv=w.Hkv, d=w.d,
                                    kv_scale=x["kv_scale"])
    assert np.max(np.abs(full - onl)) <= 1e-12


def _sdpa_reference(w, x):
    """Masked GQA attention through torch's fp64 scaled_dot_product_attention, with the
    mask built from the reading 'window row i sees keys 0..T+i' and K/V head h // G."""
    q = torch.from_numpy(_decode_bf16(x["q"]))
    if x["k"].dtype == np.uint8:
        dec = lambda c: torch.from_numpy(c).view(torch.float8_e4m3fn).to(torch.float64)
        sk = torch.from_numpy(x["kv_scale"].astype(np.float64))
        k = dec(x["k"]) * sk[0][None, :, None]
        v = dec(x["v"]) * sk[1][None, :, None]
    else:
        k = torch.from_numpy(_decode_bf16(x["k"]))
        v = torch.from_numpy(_decode_bf16(x["v"]))
    outs = []
    qo = ko = 0
    for T, D in zip(x["seq_lens"].tolist(), x["draft_len"].tolist()):
        W = D + 1
        qb = q[qo:qo + W].permute(1, 0, 2)                     # [Hq, W, d]
        kb = k[ko:ko + T + W].permute(1, 0, 2).repeat_interleave(w.G, dim=0)
        vb = v[ko:ko + T + W].permute(1, 0, 2).repeat_interleave(w.G, dim=0)
        j = torch.arange(T + W)[None, :]
        i = torch.arange(W)[:, None]
        mask = j <= T + i
        o = torch.nn.functional.scaled_dot_product_attention(qb, kb, vb, attn_mask=mask)
        outs.append(o.permute(1, 0, 2))
        qo += W
        ko += T + W
    return torch.cat(outs).numpy()


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
@pytest.mark.parametrize("shape", [
    dict(B=1, Hq=4, Hkv=1, d=64, T=(256,), D=(3,)),         # tiny-config shape, MQA
    dict(B=3, Hq=8, Hkv=2, d=32, T=(1, 17, 40), D=(4, 0, 9)),
    dict(B=2, Hq=6, Hkv=6, d=16, T=(0, 5), D=(2, 1)),       # G = 1, empty prefix
])
def test_matches_library_attention(kv, shape):
    w, x = _small(kv=kv, seed=3, **shape)
    ref = _sdpa_reference(w, x)
    got = _run(w, x)
    assert np.max(np.abs(got - ref)) <= 1e-12


def test_draft_len_zero_is_plain_decode():
    """D = 0: the single query attends to all T+1 cached keys, i.e. ordinary decode
    attention (torch SDPA without a mask)."""
    w, x = _small(B=2, Hq=8, Hkv=2, d=64, T=(100, 7), D=(0, 0), seed=4)
    got = _run(w, x)
    q = torch.from_numpy(_decode_bf16(x["q"]))
    k = torch.from_numpy(_decode_bf16(x["k"]))
    v = torch.from_numpy(_decode_bf16(x["v"]))
    ko = 0
    for b, T in enumerate(x["seq_lens"].tolist()):
        qb = q[b][:, None, :]
        kb = k[ko:ko + T + 1].permute(1, 0, 2).repeat_interleave(w.G, dim=0)
        vb = v[ko:ko + T + 1].permute(1, 0, 2).repeat_interleave(w.G, dim=0)
        ref = torch.nn.functional.scaled_dot_product_attention(qb, kb, vb)[:, 0, :].numpy()
        assert np.max(np.abs(got[b] - ref)) <= 1e-12
        ko += T + 1


def test_equal_keys_give_mean_of_visible_values():
    """All keys identical -> uniform weights over the visible keys: row i averages V rows
    0..T+i. V row j carries j in column 0, so an off-by-one mask shows up."""
    B, Hq, Hkv, d, T, D = 1, 2, 1, 8, 10, 3
    W = D + 1
    q = _bits_of(np.random.default_rng(0).standard_normal((W, Hq, d)))
    k = _bits_of(np.ones((T + W, Hkv, d)) * 0.5)
    vals = np.zeros((T + W, Hkv, d), dtype=np.float32)
    vals[:, 0, 0] = np.arange(T + W)
    vals[:, 0, 1] = 1.0
    out = oracle.verify_attn(q, k, _bits_of(vals), [T], [D], Hq=Hq, Hkv=Hkv, d=d)
    for i in range(W):
        assert abs(out[i, :, 0] - (T + i) / 2.0).max() <= 1e-12  # mean of 0..T+i
        assert abs(out[i, :, 1] - 1.0).max() <= 1e-12


# ------------------------------------------------------------- sliding window

def _sdpa_window_reference(w, x, W):
    """Torch fp64 SDPA with the sliding-window mask built from the reading 'the query at
    position p sees keys p-W+1 .. p' (p = T+i for window row i)."""
    q = torch.from_numpy(_decode_bf16(x["q"]))
    if x["k"].dtype == np.uint8:
        dec = lambda c: torch.from_numpy(c).view(torch.float8_e4m3fn).to(torch.float64)
        sk = torch.from_numpy(x["kv_scale"].astype(np.float64))
        k = dec(x["k"]) * sk[0][None, :, None]
        v = dec(x["v"]) * sk[1][None, :, None]
    else:
        k = torch.from_numpy(_decode_bf16(x["k"]))
        v = torch.from_numpy(_decode_bf16(x["v"]))
    outs = []
    qo = ko = 0
    for T, D in zip(x["seq_lens"].tolist(), x["draft_len"].tolist()):
        R = D + 1
        qb = q[qo:qo + R].permute(1, 0, 2)
        kb = k[ko:ko + T + R].permute(1, 0, 2).repeat_interleave(w.G, dim=0)
        vb = v[ko:ko + T + R].permute(1, 0, 2).repeat_interleave(w.G, dim=0)
        j = torch.arange(T + R)[None, :]
        p = T + torch.arange(R)[:, None]
        mask = (j <= p) & (j > p - W)
        o = torch.nn.functional.scaled_dot_product_attention(qb, kb, vb, attn_mask=mask)
        outs.append(o.permute(1, 0, 2))
        qo += R
        ko += T + R
    return torch.cat(outs).numpy()


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
@pytest.mark.parametrize("W", [1, 2, 5, 16, 41, 1000])
def test_sliding_window_matches_library_attention(kv, W):
    w, x = _small(B=3, Hq=8, Hkv=2, d=32, T=(1, 17, 40), D=(4, 0, 9), seed=7, kv=kv)
    ref = _sdpa_window_reference(w, x, W)
    got = _run(w, x, window=W)
    assert np.max(np.abs(got - ref)) <= 1e-12


def test_sliding_window_equal_keys_give_mean_of_last_w_values():
    """All keys identical -> uniform weights over the window: row i averages V rows
    max(0, T+i-W+1) .. T+i. V row j carries j in column 0, so an off-by-one lower or
    upper bound changes the mean."""
    Hq, Hkv, d, T, D = 2, 1, 8, 10, 3
    R = D + 1
    q = _bits_of(np.random.default_rng(0).standard_normal((R, Hq, d)))
    k = _bits_of(np.ones((T + R, Hkv, d)) * 0.5)
    vals = np.zeros((T + R, Hkv, d), dtype=np.float32)
    vals[:, 0, 0] = np.arange(T + R)
    vals[:, 0, 1] = 1.0
    for W in (1, 2, 3, 7, 11, 12, 13, 14, 50):
        out = oracle.verify_attn(q, k, _bits_of(vals), [T], [D], Hq=Hq, Hkv=Hkv, d=d,
                                 window=W)
        for i in range(R):
            lo = max(0, T + i - W + 1)
            assert abs(out[i, :, 0] - (lo + T + i) / 2.0).max() <= 1e-12
            assert abs(out[i, :, 1] - 1.0).max() <= 1e-12


def test_window_of_one_returns_the_rows_own_value():
    """W = 1: each query sees only its own position, so the output is that V row."""
    w, x = _small(B=2, Hq=4, Hkv=2, d=16, T=(5, 0), D=(3, 2), seed=8)
    got = _run(w, x, window=1)
    v = _decode_bf16(x["v"])
    qo = ko = 0
    for T, D in zip(x["seq_lens"].tolist(), x["draft_len"].tolist()):
        for i in range(D + 1):
            for h in range(w.Hq):
                assert np.array_equal(got[qo + i, h], v[ko + T + i, h // w.G])
        qo += D + 1
        ko += T + D + 1


def test_window_covering_every_key_is_full_attention():
    """W >= T+D+1 keeps every key: the result equals the unwindowed one exactly."""
    w, x = _small(B=2, Hq=4, Hkv=1, d=16, T=(6, 12), D=(2, 5), seed=9)
    full = _run(w, x)
    for W in (18, 19, 10 ** 6):
        assert np.array_equal(_run(w, x, window=W), full)
    assert not np.array_equal(_run(w, x, window=17), full)  # the last row loses key 0


@pytest.mark.parametrize("tile", [1, 4, 7])
def test_sliding_window_online_equals_materialised(tile):
    w, x = _small(B=3, Hq=8, Hkv=2, d=32, T=(1, 17, 40), D=(4, 0, 9), seed=10)
    for W in (3, 9, 30):
        a = _run(w, x, window=W)
        b = _run(w, x, window=W, online_tile=tile)
        assert np.max(np.abs(a - b)) <= 1e-12


def test_sliding_window_never_reads_positions_before_it():
    """Cache rows of positions before T-W+1 are outside every row's window: NaN there
    leaves every output finite and unchanged."""
    w, x = _small(B=2, Hq=4, Hkv=2, d=16, T=(30, 22), D=(3, 6), seed=11)
    W = 8
    ref = _run(w, x, window=W)
    k, v = x["k"].copy(), x["v"].copy()
    ko = 0
    for T, D in zip(x["seq_lens"].tolist(), x["draft_len"].tolist()):
        k[ko:ko + T - W + 1] = 0x7FC0  # bf16 NaN
        v[ko:ko + T - W + 1] = 0x7FC0
        ko += T + D + 1
    got = _run(w, dict(x, k=k, v=v), window=W)
    assert np.isfinite(got).all() and np.array_equal(got, ref)


# ------------------------------------------------------------------- paged cache

def _paged_oracle(w, x, pg, **kw):
    return oracle.verify_attn_paged(x["q"], pg["k_pages"], pg["v_pages"], pg["block_table"],
                                    x["seq_lens"], x["draft_len"], Hq=w.Hq, Hkv=w.Hkv, d=w.d,
                                    kv_scale=x["kv_scale"], **kw)


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
@pytest.mark.parametrize("bs", [1, 4, 16, 64])
def test_paged_equals_packed_for_any_block_placement(kv, bs):
    """Blocks at random physical slots among NaN-filled spares give exactly the packed
    result: every position is found through the table and nothing else is read."""
    w, x = _small(B=3, Hq=8, Hkv=2, d=32, T=(1, 17, 40), D=(4, 0, 9), seed=12, kv=kv)
    pg = synth.paged_layout(x, bs, seed=5, spare_blocks=4)
    assert np.array_equal(_paged_oracle(w, x, pg), _run(w, x))


def test_paged_brute_force_walk_of_the_block_table():
    """One output row recomputed in numpy by walking the block table position by position
    (softmax over the fetched keys, weighted sum of the fetched values)."""
    w, x = _small(B=2, Hq=4, Hkv=2, d=16, T=(23, 9), D=(3, 2), seed=13)
    bs = 8
    pg = synth.paged_layout(x, bs, seed=6, spare_blocks=2)
    got = _paged_oracle(w, x, pg)
    kp = _decode_bf16(pg["k_pages"])
    vp = _decode_bf16(pg["v_pages"])
    q = _decode_bf16(x["q"])
    qo = 0
    for b, (T, D) in enumerate(zip(x["seq_lens"].tolist(), x["draft_len"].tolist())):
        for i in range(D + 1):
            for h in range(w.Hq):
                g = h // w.G
                keys = [kp[pg["block_table"][b, j // bs], j % bs, g] for j in range(T + i + 1)]
                vals = [vp[pg["block_table"][b, j // bs], j % bs, g] for j in range(T + i + 1)]
                s_ = np.array([q[qo + i, h] @ kk for kk in keys]) / math.sqrt(w.d)
                p_ = np.exp(s_ - s_.max())
                ref = (p_ / p_.sum()) @ np.array(vals)
                assert np.max(np.abs(got[qo + i, h] - ref)) <= 1e-12
        qo += D + 1


@pytest.mark.parametrize("bs", [4, 16])
def test_paged_with_window_and_reclaimed_blocks(bs):
    """Blocks wholly before every row's sliding window handed back to the pool (table
    entries -1, slots NaN): the windowed result equals the packed windowed one."""
    w, x = _small(B=3, Hq=8, Hkv=2, d=32, T=(70, 17, 45), D=(4, 0, 9), seed=14)
    W = 20
    pg = synth.paged_layout(x, bs, seed=7, spare_blocks=2, reclaim_before_window=W)
    assert (pg["block_table"][0, :2] == -1).all()  # positions 0..7 of sequence 0 are gone
    assert np.array_equal(_paged_oracle(w, x, pg, window=W), _run(w, x, window=W))


def test_constant_values_per_kv_head_select_the_group():
    """V constant per KV head -> every query head h returns its group's constant c[h//G]."""
    B, Hq, Hkv, d, T, D = 2, 8, 4, 16, 6, 2
    rng = np.random.default_rng(5)
    n_kv = B * (T + D + 1)
    q = _bits_of(rng.standard_normal((B * (D + 1), Hq, d)))
    k = _bits_of(rng.standard_normal((n_kv, Hkv, d)))
    c = np.array([1.0, -2.0, 3.5, 0.25], dtype=np.float32)
    v = _bits_of(np.broadcast_to(c[None, :, None], (n_kv, Hkv, d)))
    out = oracle.verify_attn(q, k, v, [T] * B, [D] * B, Hq=Hq, Hkv=Hkv, d=d)
    expect = np.repeat(c, Hq // Hkv)[None, :, None]
    assert np.max(np.abs(out - expect)) <= 1e-12


def test_dominant_key_returns_its_value():
    """One key with a score far above the rest -> that key's V row (weight 1 - O(e^-100))."""
    Hq, Hkv, d, T, D = 1, 1, 16, 12, 1
    q = np.zeros((D + 1, Hq, d), dtype=np.float32)
    q[:, 0, 0] = 64.0
    k = np.zeros((T + D + 1, Hkv, d), dtype=np.float32)
    k[5, 0, 0] = 16.0                         # score 64*16/4 = 256 vs 0 elsewhere
    v = np.random.default_rng(6).standard_normal((T + D + 1, Hkv, d)).astype(np.float32)
    vb = _bits_of(v)
    out = oracle.verify_attn(_bits_of(q), _bits_of(k), vb, [T], [D], Hq=Hq, Hkv=Hkv, d=d)
    assert np.max(np.abs(out[:, 0, :] - _decode_bf16(vb)[5, 0][None, :])) <= 1e-12


def test_two_keys_logistic_weights_and_scale():
    """T = 0, D = 1: row 0 sees one key (output = v0); row 1 sees two keys with scores
    s0, s1 = q.k * scale and returns sigma(s0 - s1) v0 + sigma(s1 - s0) v1. Default scale
    is 1/sqrt(d); an explicit scale overrides it."""
    d = 4
    q = _bits_of(np.array([[[1.0, 0, 0, 0]], [[1.0, 0.5, 0, 0]]]))
    k = _bits_of(np.array([[[2.0, 0, 0, 0]], [[0.0, 3.0, 0, 0]]]))
    v = _bits_of(np.array([[[1.0, 0, 0, 0]], [[0, 1.0, 0, 0]]]))
    for scale in (None, 0.3):
        out = oracle.verify_attn(q, k, v, [0], [1], Hq=1, Hkv=1, d=d, scale=scale)
        sc = 1 / math.sqrt(d) if scale is None else scale
        s0, s1 = 2.0 * sc, 1.5 * sc
        w0 = 1 / (1 + math.exp(s1 - s0))
        assert np.max(np.abs(out[0, 0] - [1, 0, 0, 0])) <= 1e-15
        assert abs(out[1, 0, 0] - w0) <= 1e-15 and abs(out[1, 0, 1] - (1 - w0)) <= 1e-15


def test_prefix_permutation_invariance():
    """Permuting the cached-prefix slots (same permutation for K and V) changes nothing;
    the window slots keep their order because the mask depends on it."""
    w, x = _small(B=2, Hq=8, Hkv=2, d=32, T=(50, 20), D=(6, 3), seed=7)
    base = _run(w, x)
    rng = np.random.default_rng(8)
    k, v = x["k"].copy(), x["v"].copy()
    ko = 0
    for T, D in zip(x["seq_lens"].tolist(), x["draft_len"].tolist()):
        perm = ko + rng.permutation(T)
        k[ko:ko + T] = x["k"][perm]
        v[ko:ko + T] = x["v"][perm]
        ko += T + D + 1
    got = oracle.verify_attn(x["q"], k, v, x["seq_lens"], x["draft_len"], Hq=w.Hq,
                             Hkv=w.Hkv, d=w.d)
    assert np.max(np.abs(got - base)) <= 1e-12
    # a window slot swap does change the result (the mask sees positions)
    k2 = x["k"].copy()
    T0 = int(x["seq_lens"][0])
    k2[[T0, T0 + 3]] = k2[[T0 + 3, T0]]
    moved = oracle.verify_attn(x["q"], k2, x["v"], x["seq_lens"], x["draft_len"], Hq=w.Hq,
                               Hkv=w.Hkv, d=w.d)
    assert np.max(np.abs(moved - base)) > 1e-6


def test_fp8_scales_act_on_scores_and_values():
    """K scale multiplies the scores (same as multiplying the softmax scale); V scale
    multiplies the output linearly."""
    w, x = _small(kv="fp8_e4m3", B=2, Hq=4, Hkv=2, d=32, T=(30, 9), D=(3, 2), seed=9)
    base = _run(w, x)
    sc = x["kv_scale"].copy()
    sc[0] *= 2.0
    sc[1] *= 4.0  # powers of two keep the fp32 scales exact
    got = oracle.verify_attn(x["q"], x["k"], x["v"], x["seq_lens"], x["draft_len"],
                             Hq=w.Hq, Hkv=w.Hkv, d=w.d, kv_scale=sc,
                             scale=2.0 / math.sqrt(w.d))
    ref = 4.0 * oracle.verify_attn(x["q"], x["k"], x["v"], x["seq_lens"], x["draft_len"],
                                   Hq=w.Hq, Hkv=w.Hkv, d=w.d, kv_scale=x["kv_scale"],
                                   scale=4.0 / math.sqrt(w.d))
    assert np.max(np.abs(got - ref)) <= 1e-12
    assert np.max(np.abs(base - got / 4.0)) > 1e-6


def test_unit_mask_computes_only_selected_units():
    w, x = _small(B=2, Hq=4, Hkv=2, d=16, T=(9, 4), D=(1, 2), seed=10)
    full = _run(w, x)
    part = _run(w, x, units=[(1, 0)])
    G = w.G
    assert np.array_equal(part[2:5, 0:G], full[2:5, 0:G])
    assert np.isnan(part[0:2]).all() and np.isnan(part[2:5, G:]).all()


# ---------------------------------------------------------------- acceptance

def _read_worked_examples():
    rows = []
    with open(os.path.join(GOLDEN, "worked_example_accept.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            name, draft, tgt, al, nt = [s.strip() for s in line.split("|")]
            rows.append((name, [int(t) for t in draft.split()], [int(t) for t in tgt.split()],
                         int(al), int(nt)))
    return rows


@pytest.mark.parametrize("case", _read_worked_examples(), ids=lambda c: c[0])
def test_worked_acceptance_example(case):
    _, draft, tgt, al, nt = case
    V = 64
    logits = np.random.default_rng(11).standard_normal((len(tgt), V)).astype(np.float32)
    for r, t in enumerate(tgt):
        logits[r, t] = 10.0
    got_al, got_nt, amax = oracle.spec_accept(logits, np.array(draft), np.array([len(draft)]))
    assert list(amax) == tgt
    assert got_al[0] == al and got_nt[0] == nt


def test_argmax_lowest_index_tie_break():
    V = 100
    logits = np.zeros((4, V), dtype=np.float32)
    logits[0, [7, 30, 99]] = 2.0              # plain three-way tie -> 7
    logits[1, :] = -1.0                        # all equal -> 0
    logits[2, 50] = -0.0
    logits[2, :] = -3.0
    logits[2, [50, 60]] = [0.0, -0.0]          # +0 and -0 tie -> 50
    logits[2, 40] = -0.0                       # -0 earlier -> 40
    logits[3, [98, 99]] = 1.0                  # tie at the tail
    amax = oracle.argmax_rows(logits)
    assert list(amax) == [7, 0, 40, 98]
    bits = synth.bf16_bits(logits)
    assert list(oracle.argmax_rows(bits)) == [7, 0, 40, 98]


def test_argmax_matches_numpy_first_occurrence_on_tied_bf16():
    """bf16-rounded N(0,1) rows over a large vocab share their maximum often; numpy's
    argmax is documented to return the first occurrence."""
    rng = np.random.default_rng(12)
    bits = synth.bf16_bits(rng.standard_normal((256, 128256)).astype(np.float32))
    vals = _decode_bf16(bits)
    ties = sum(int((r == r.max()).sum() > 1) for r in vals)
    assert ties >= 3
    assert np.array_equal(oracle.argmax_rows(bits), np.argmax(vals, axis=1))


def test_acceptance_length_range():
    """1 <= AL <= 1 + D for every sequence; next_token is the target's token at row AL-1."""
    for seed in range(5):
        w = synth.CONFIGS["c5"].with_(V=50, B=64)
        a = synth.accept_inputs(w, seed)
        al, nt, amax = oracle.spec_accept(a["logits"], a["draft_tokens"], a["draft_len"])
        D = a["draft_len"]
        assert np.all(al >= 1) and np.all(al <= D + 1)
        q_off = np.concatenate([[0], np.cumsum(D + 1)])[:-1]
        assert np.array_equal(nt, amax[q_off + al - 1])


def _golden_al():
    out = []
    with open(os.path.join(GOLDEN, "expected_al_k4.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            a, k, v, dec = line.split()
            out.append((float(a), int(k), float(v), int(dec)))
    return out


@pytest.mark.parametrize("alpha,k,printed,dec", _golden_al())
def test_expected_acceptance_length(alpha, k, printed, dec):
    """Mean AL over many sequences whose drafts match independently with probability
    alpha equals (1 - alpha^(k+1)) / (1 - alpha) within 4 sigma; that closed form rounds
    to the page's printed value."""
    closed = k + 1.0 if alpha == 1.0 else (1 - alpha ** (k + 1)) / (1 - alpha)
    assert round(closed, dec) == printed
    n = 6000
    w = synth.Workload("al", B=n, Hq=1, Hkv=1, d=8, D=k, T=1, V=32, p=alpha,
                       logits_dtype="fp32")
    a = synth.accept_inputs(w, 13)
    al, _, _ = oracle.spec_accept(a["logits"], a["draft_tokens"], a["draft_len"])
    # variance of AL = 1 + (leading matches)
    pmf = np.array([alpha ** j * (1 - alpha) for j in range(k)] + [alpha ** k])
    vals = np.arange(1, k + 2)
    var = float(np.sum(pmf * vals ** 2) - np.sum(pmf * vals) ** 2)
    assert abs(al.mean() - closed) <= 4 * math.sqrt(var / n) + 1e-12


def test_accept_rejects_bad_sizes():
    with pytest.raises(ValueError):
        oracle.accept(np.zeros(3, np.int32), np.zeros(3, np.int32), np.array([3]))


# ------------------------------------------------------------------ draft signals

def test_draft_signals_uniform_and_equal_maxima():
    """Equal logits: confidence 1/V, entropy ln V. k equal maxima with the rest at -inf:
    confidence 1/k, entropy ln k."""
    V = 1000
    conf, ent = oracle.draft_signals(np.full((2, V), 0.25, dtype=np.float32))
    assert np.allclose(conf, 1.0 / V, rtol=1e-12) and np.allclose(ent, math.log(V), rtol=1e-12)
    for k in (1, 2, 7):
        x = np.full((1, V), -np.inf, dtype=np.float32)
        x[0, np.arange(k) * 97] = 3.0
        conf, ent = oracle.draft_signals(x)
        assert conf[0] == pytest.approx(1.0 / k, rel=1e-12)
        assert ent[0] == pytest.approx(math.log(k), abs=1e-12)


@pytest.mark.parametrize("a", [0.0, 0.5, -3.0, 12.0])
def test_draft_signals_two_point_closed_form(a):
    """Two finite logits (a, 0), the rest -inf: p = 1/(1 + e^-a); confidence max(p, 1-p),
    entropy -p ln p - (1-p) ln(1-p)."""
    x = np.full((1, 50), -np.inf, dtype=np.float32)
    x[0, 3], x[0, 40] = a, 0.0
    p = 1.0 / (1.0 + math.exp(-a))
    conf, ent = oracle.draft_signals(x)
    assert conf[0] == pytest.approx(max(p, 1 - p), rel=1e-12)
    h = -p * math.log(p) - (1 - p) * math.log(1 - p)
    assert ent[0] == pytest.approx(h, rel=1e-10, abs=1e-15)


def test_draft_signals_match_library_softmax_entropy():
    """Random rows against scipy's softmax and entropy (natural log), fp32 and bf16."""
    scipy_special = pytest.importorskip("scipy.special")
    scipy_stats = pytest.importorskip("scipy.stats")
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((6, 3001)) * rng.uniform(0.1, 6.0, (6, 1))).astype(np.float32)
    for logits, vals in ((x, x.astype(np.float64)),
                         (synth.bf16_bits(x), None)):
        if vals is None:
            vals = (logits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        conf, ent = oracle.draft_signals(logits)
        p = scipy_special.softmax(vals, axis=1)
        assert np.allclose(conf, p.max(axis=1), rtol=1e-12)
        assert np.allclose(ent, scipy_stats.entropy(p, axis=1), rtol=1e-10)


def test_draft_signals_shift_invariance_and_bounds():
    """Adding a constant to a row changes neither signal; 1/V <= confidence <= 1,
    0 <= entropy <= ln V, and confidence >= exp(-entropy) (min-entropy <= entropy)."""
    rng = np.random.default_rng(6)
    V = 777
    x = (rng.standard_normal((8, V)) * 3).astype(np.float32)
    c0, h0 = oracle.draft_signals(x)
    c1, h1 = oracle.draft_signals(x + np.float32(17.0))
    assert np.allclose(c0, c1, rtol=1e-5) and np.allclose(h0, h1, rtol=1e-5, atol=1e-6)
    assert np.all(c0 >= 1.0 / V) and np.all(c0 <= 1.0)
    assert np.all(h0 >= 0) and np.all(h0 <= math.log(V) + 1e-12)
    assert np.all(c0 >= np.exp(-h0) - 1e-12)
