"""Pins of the oracle's stochastic (distribution-preserving) acceptance against what the
pages and the mathematics fix, not against its own formula.

"GPU and LLM, chapter 5", "Speculative decoding (2)": the acceptance rule leaves the
distribution of the output exactly that of the large model alone. So, with drafts drawn
from the drafter's distribution q and uniform draws, every emitted token must follow the
target's softmax p of its row: the first token p_0, the second (given the first draft was
kept) p_1, and the bonus token after all D drafts p_D. The probability of keeping a draft
is sum_x min(p(x), q(x)). Closed forms: q = p keeps every draft; a drafter certain of x
where the target gives x probability 0 is always rejected, and the token drawn then
follows p without x; D = 0 draws straight from p_0. CPU only."""
import numpy as np
import pytest

import oracle


def _softmax(x):
    z = np.exp(x - x.max())
    return z / z.sum()


def _within(freq, prob, n, k=4.5):
    sigma = np.sqrt(np.maximum(prob * (1 - prob), 1e-12) / n)
    return np.all(np.abs(freq - prob) <= k * sigma + 1e-12), np.max(np.abs(freq - prob) / sigma)


@pytest.mark.parametrize("temperature", [1.0, 0.6])
def test_emitted_tokens_follow_the_target_distribution(temperature):
    rng = np.random.default_rng(11)
    V, D, N = 6, 2, 40000
    tgt = (rng.standard_normal((D + 1, V)) * 1.5).astype(np.float32)
    drf = (tgt[:D] + rng.standard_normal((D, V)) * 1.2).astype(np.float32)
    p = [_softmax(tgt[j].astype(np.float64) / temperature) for j in range(D + 1)]
    q = [_softmax(drf[j].astype(np.float64) / temperature) for j in range(D)]
    # N sequences with the same rows; the drafter samples its tokens from q
    toks = np.stack([rng.choice(V, size=N, p=q[j]) for j in range(D)], axis=1).astype(np.int32)
    al, nt, ma, ms = oracle.accept_stochastic(
        np.tile(tgt, (N, 1)), np.tile(drf, (N, 1)), toks.reshape(-1), np.full(N, D, np.int32),
        rng.random(N * D, dtype=np.float32), rng.random(N, dtype=np.float32), temperature)
    assert np.all((al >= 1) & (al <= D + 1))
    assert np.all((ma >= 0) & (ma <= 1)) and np.all((ms >= 0) & (ms <= 0.5))
    first = np.where(al >= 2, toks[:, 0], nt)
    ok, z = _within(np.bincount(first, minlength=V) / N, p[0], N)
    assert ok, z
    kept0 = al >= 2
    ok, z = _within(np.array([kept0.mean()]), np.array([np.minimum(p[0], q[0]).sum()]), N)
    assert ok, z
    second = np.where(al[kept0] >= 3, toks[kept0, 1], nt[kept0])
    n2 = int(kept0.sum())
    ok, z = _within(np.bincount(second, minlength=V) / n2, p[1], n2)
    assert ok, z
    bonus = nt[al == D + 1]
    ok, z = _within(np.bincount(bonus, minlength=V) / len(bonus), p[D], len(bonus))
    assert ok, z


def _inverse_cdf(w, u):
    """numpy's searchsorted on the running sums: the first index whose running sum exceeds
    u times the total."""
    c = np.cumsum(w)
    return int(np.searchsorted(c, u * c[-1], side="right"))


def test_draft_equal_to_target_keeps_every_draft():
    rng = np.random.default_rng(3)
    B, D, V = 50, 4, 300
    tgt = rng.standard_normal((B * (D + 1), V)).astype(np.float32)
    drf = np.concatenate([tgt[b * (D + 1):b * (D + 1) + D] for b in range(B)])
    toks = rng.integers(0, V, size=B * D).astype(np.int32)
    us = rng.random(B, dtype=np.float32)
    al, nt, _, _ = oracle.accept_stochastic(tgt, drf, toks, np.full(B, D, np.int32),
                                         rng.random(B * D, dtype=np.float32), us)
    assert np.all(al == D + 1)
    for b in range(B):
        pD = _softmax(tgt[b * (D + 1) + D].astype(np.float64))
        assert nt[b] == _inverse_cdf(pD, float(us[b]))


def test_certain_drafter_on_an_impossible_token_is_rejected():
    """q one-hot at x (its logit far above the rest) and p(x) = 0: the draft is never kept,
    and the residual max(0, p - q) is p with x removed."""
    rng = np.random.default_rng(4)
    V, B = 50, 40
    tgt = rng.standard_normal((2 * B, V)).astype(np.float32)
    drf = np.full((B, V), -1e30, dtype=np.float32)
    x = rng.integers(0, V, size=B).astype(np.int32)
    for b in range(B):
        tgt[2 * b, x[b]] = -np.inf
        drf[b, x[b]] = 0.0
    us = rng.random(B, dtype=np.float32)
    al, nt, _, _ = oracle.accept_stochastic(tgt, drf, x, np.ones(B, np.int32),
                                         rng.random(B, dtype=np.float32), us)
    assert np.all(al == 1)
    for b in range(B):
        w = _softmax(tgt[2 * b].astype(np.float64))
        w[x[b]] = 0.0
        assert nt[b] == _inverse_cdf(w, float(us[b])) and nt[b] != x[b]


def test_no_drafts_draws_from_the_first_row():
    rng = np.random.default_rng(5)
    B, V = 30, 1000
    tgt = rng.standard_normal((B, V)).astype(np.float32)
    us = rng.random(B, dtype=np.float32)
    al, nt, _, _ = oracle.accept_stochastic(tgt, np.zeros((0, V), np.float32),
                                         np.zeros(0, np.int32), np.zeros(B, np.int32),
                                         np.zeros(0, np.float32), us)
    assert np.all(al == 1)
    assert all(nt[b] == _inverse_cdf(_softmax(tgt[b].astype(np.float64)), float(us[b]))
               for b in range(B))


def test_temperature_divides_the_logits():
    rng = np.random.default_rng(6)
    B, D, V = 20, 3, 200
    tgt = rng.standard_normal((B * (D + 1), V)).astype(np.float32)
    drf = rng.standard_normal((B * D, V)).astype(np.float32)
    toks = rng.integers(0, V, size=B * D).astype(np.int32)
    ua, us = rng.random(B * D, dtype=np.float32), rng.random(B, dtype=np.float32)
    Dv = np.full(B, D, np.int32)
    a = oracle.accept_stochastic(tgt, drf, toks, Dv, ua, us, temperature=2.0)
    b = oracle.accept_stochastic(tgt * np.float32(0.5), drf * np.float32(0.5), toks, Dv, ua, us)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_bf16_logits_decode_like_fp32():
    from speculative_decoding_verification_gqa_gb300 import synth
    rng = np.random.default_rng(7)
    B, D, V = 10, 2, 333
    tgt = synth.bf16_bits(rng.standard_normal((B * (D + 1), V)).astype(np.float32))
    drf = synth.bf16_bits(rng.standard_normal((B * D, V)).astype(np.float32))
    widen = lambda b: (b.astype(np.uint32) << np.uint32(16)).view(np.float32)
    toks = rng.integers(0, V, size=B * D).astype(np.int32)
    ua, us = rng.random(B * D, dtype=np.float32), rng.random(B, dtype=np.float32)
    Dv = np.full(B, D, np.int32)
    a = oracle.accept_stochastic(tgt, drf, toks, Dv, ua, us)
    b = oracle.accept_stochastic(widen(tgt), widen(drf), toks, Dv, ua, us)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))


def test_mean_acceptance_length_matches_the_printed_values():
    """With two-token distributions p = (a, 1 - a) and q = (b, 1 - b) at every draft
    position, a draft drawn from q is kept with probability alpha = 1 - |a - b|,
    independently of the other positions. So the mean acceptance length of k = 4 drafts is
    (1 - alpha^5) / (1 - alpha), the expected value the pages print for alpha = 0.5, 0.7
    and 0.9 (tests/golden/expected_al_k4.txt; alpha = 1 gives k + 1)."""
    import os
    golden = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                          "expected_al_k4.txt")
    rows = [l.split() for l in open(golden) if l.strip() and not l.startswith("#")]
    rng = np.random.default_rng(12)
    N = 30000
    for alpha_s, k_s, printed_s, decimals_s in rows:
        alpha, k, printed = float(alpha_s), int(k_s), float(printed_s)
        a = 0.9
        b = a - (1.0 - alpha)  # |a - b| = 1 - alpha
        lt = np.log(np.array([a, 1 - a]))
        ld = np.log(np.array([max(b, 1e-300), 1 - b]))
        tgt = np.tile(lt, (N * (k + 1), 1)).astype(np.float32)
        drf = np.tile(ld, (N * k, 1)).astype(np.float32)
        toks = (rng.random(N * k) >= b).astype(np.int32)  # token 0 with probability b
        al, _, _, _ = oracle.accept_stochastic(tgt, drf, toks, np.full(N, k, np.int32),
                                               rng.random(N * k, dtype=np.float32),
                                               rng.random(N, dtype=np.float32))
        exact = (1 - alpha ** (k + 1)) / (1 - alpha) if alpha < 1 else k + 1.0
        assert round(exact, int(decimals_s)) == printed
        sigma = al.std() / np.sqrt(N) + 1e-12
        assert abs(al.mean() - exact) <= 4.5 * sigma + 1e-9, (alpha, al.mean(), exact)
