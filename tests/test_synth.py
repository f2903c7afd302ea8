"""Input generator checks (CPU): rounding, determinism, recipe statistics."""
import numpy as np
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
