"""Input generator checks (CPU): rounding, determinism, recipe statistics."""
import numpy as np
import pytest
import torch

from speculative_decoding_verification_gqa_gb300 import synth


def test_bf16_rounding_matches_torch():
    x = np.random.default_rng(0).standard_normal(100000).astype(np.float32) * 7
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(synth.bf16_bits(x), ref)


def test_deterministic_and_seed_sensitive():
    w = synth.CONFIGS["c1"]
    a = synth.attn_inputs(w, 5)
    b = synth.attn_inputs(w, 5)
    c = synth.attn_inputs(w, 6)
    assert np.array_equal(a["k"], b["k"]) and not np.array_equal(a["k"], c["k"])
    assert a["q"].shape == (4, 4, 64) and a["k"].shape == (260, 1, 64)


def test_fp8_recipe_scales_and_range():
    w = synth.CONFIGS["c3"].with_(B=2, T=300, D=3)
    x = synth.attn_inputs(w, 1)
    assert x["k"].dtype == np.uint8 and x["kv_scale"].shape == (2, w.Hkv)
    dec = torch.from_numpy(x["k"]).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    # absmax per head maps to the top code 448
    assert np.allclose(np.abs(dec).max(axis=(0, 2)), 448.0)
    assert not np.isnan(dec).any()


def test_ragged_lengths_recipe():
    T, D, p = synth.lengths(synth.CONFIGS["c5"], 0)
    assert T.min() >= 1024 and T.max() <= 65536 and set(D.tolist()) <= {1, 2, 4, 8}
    assert p.min() > 0.4 and p.max() < 0.9


def test_draft_match_rate():
    w = synth.Workload("m", B=4000, Hq=1, Hkv=1, d=8, D=3, T=1, V=40, p=0.7,
                       logits_dtype="fp32")
    a = synth.accept_inputs(w, 2)
    greedy = np.argmax(a["logits"], axis=1).reshape(4000, 4)[:, :3].reshape(-1)
    rate = np.mean(greedy == a["draft_tokens"])
    assert abs(rate - 0.7) < 0.02
    assert a["draft_tokens"].min() >= 0 and a["draft_tokens"].max() < 40


def _paged_case(bs, reclaim=0, spare=3, kv="bf16"):
    w = synth.Workload("p", B=4, Hq=4, Hkv=2, d=16, D=0, T=0, V=8, p=0.5, kv_dtype=kv)
    x = synth.attn_inputs(w, 3, seq_lens=np.array([0, 37, 100, 5]),
                          draft_len=np.array([4, 0, 7, 2]))
    return x, synth.paged_layout(x, bs, seed=9, spare_blocks=spare, reclaim_before_window=reclaim)


def test_paged_layout_round_trips_every_position():
    """Position j of sequence b sits at row j % bs of block table[b, j // bs], blocks are
    distinct and inside the pool, entries past a sequence's last block are -1, and unused
    rows hold the NaN fill."""
    for bs in (1, 4, 16, 64):
        x, pg = _paged_case(bs)
        kp, tab = pg["k_pages"], pg["block_table"]
        T = x["seq_lens"].astype(int)
        R = T + x["draft_len"].astype(int) + 1
        used = []
        row0 = 0
        for b in range(len(T)):
            nblk = -(-R[b] // bs)
            assert (tab[b, nblk:] == -1).all()
            used += list(tab[b, :nblk])
            for j in range(R[b]):
                assert np.array_equal(kp[tab[b, j // bs], j % bs], x["k"][row0 + j])
                assert np.array_equal(pg["v_pages"][tab[b, j // bs], j % bs], x["v"][row0 + j])
            if R[b] % bs:
                assert (kp[tab[b, nblk - 1], R[b] % bs:] == 0x7FC0).all()
            row0 += R[b]
        assert len(set(used)) == len(used)
        assert min(used) >= 0 and max(used) < kp.shape[0]
        assert kp.shape[0] == len(used) + 3


def test_paged_layout_reclaims_exactly_the_blocks_before_the_window():
    W, bs = 20, 8
    x, pg = _paged_case(bs, reclaim=W)
    tab = pg["block_table"]
    T = x["seq_lens"].astype(int)
    for b in range(len(T)):
        first_kept = max(T[b] - W + 1, 0) // bs  # blocks holding only earlier positions
        assert (tab[b, :first_kept] == -1).all()
        R = T[b] + int(x["draft_len"][b]) + 1
        assert (tab[b, first_kept:-(-R // bs)] >= 0).all()


def test_paged_layout_fp8_fill_is_the_e4m3_nan_code():
    x, pg = _paged_case(16, kv="fp8_e4m3")
    kp, tab = pg["k_pages"], pg["block_table"]
    spare = sorted(set(range(kp.shape[0])) - set(tab[tab >= 0].tolist()))
    assert len(spare) == 3 and (kp[spare] == 0x7F).all()


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_stochastic_inputs_recipe(dtype):
    w = synth.Workload("s", B=6, Hq=1, Hkv=1, d=8, D=5, T=1, V=777, p=0.8, logits_dtype=dtype)
    Dv = np.array([5, 0, 3, 5, 1, 2], dtype=np.int32)
    x = synth.stochastic_inputs(w, 9, draft_len=Dv, noise=0.25)
    y = synth.stochastic_inputs(w, 9, draft_len=Dv, noise=0.25)
    assert all(np.array_equal(x[k], y[k]) for k in x)
    nd = int(Dv.sum())
    assert x["target_logits"].shape == (nd + 6, 777) and x["draft_logits"].shape == (nd, 777)
    assert x["draft_logits"].dtype == x["target_logits"].dtype
    assert x["draft_tokens"].shape == (nd,) and x["draft_tokens"].min() >= 0
    assert x["draft_tokens"].max() < 777
    for u, n in ((x["u_accept"], nd), (x["u_sample"], 6)):
        assert u.dtype == np.float32 and u.shape == (n,) and u.min() >= 0 and u.max() < 1
    # the drafter's row j of sequence b is the target's row j plus N(0, 0.25^2) noise
    widen = (lambda a: (a.astype(np.uint32) << np.uint32(16)).view(np.float32)) \
        if dtype == "bf16" else (lambda a: a)
    rows = [int(np.sum(Dv[:b] + 1)) + j for b in range(6) for j in range(int(Dv[b]))]
    diff = widen(x["draft_logits"]) - widen(x["target_logits"][rows])
    assert abs(float(diff.std()) - 0.25) < 0.02 and abs(float(diff.mean())) < 0.01
    # the accept-step logits are the same as spec_accept's inputs of that seed
    a = synth.accept_inputs(w, 9, draft_len=Dv)
    assert np.array_equal(a["logits"], x["target_logits"])
