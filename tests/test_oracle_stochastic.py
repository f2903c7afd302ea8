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


def test_all_zero_residual_draws_from_the_target():
    """p = q at the draft position and the drafted token has probability 0 under both
    (logit -inf in both rows): u q(x) < p(x) reads 0 < 0, so the draft is rejected, and
    every weight of max(0, p - q) is 0. The emitted token then follows p (the output must
    keep the target's distribution): exactly numpy's inverse CDF of p at u_sample for every
    sequence, and over 40,000 sequences each token's frequency within 4.5 sigma of p."""
    rng = np.random.default_rng(21)
    V, N = 7, 40000
    row = (rng.standard_normal(V) * 1.3).astype(np.float32)
    x = 3
    row[x] = -np.inf
    p = _softmax(row.astype(np.float64))
    assert p[x] == 0.0
    tgt = np.tile(row, (2 * N, 1))            # rows 0 and 1 of every sequence
    drf = np.tile(row, (N, 1))                # q = p at the draft position
    us = rng.random(N, dtype=np.float32)
    al, nt, ma, _ = oracle.accept_stochastic(tgt, drf, np.full(N, x, np.int32),
                                             np.ones(N, np.int32),
                                             rng.random(N, dtype=np.float32), us)
    assert np.all(al == 1) and np.all(ma == 0.0)
    assert all(nt[b] == _inverse_cdf(p, float(us[b])) for b in range(0, N, 97))
    assert np.all(nt != x)
    ok, z = _within(np.bincount(nt, minlength=V) / N, p, N)
    assert ok, z


def test_all_zero_residual_after_kept_drafts():
    """The same degenerate rejection at the third draft position, after two drafts that
    q = p keeps whenever u < 1: the token is drawn from the target's row of that position,
    not from the first row or the bonus row."""
    rng = np.random.default_rng(22)
    V, B, D = 11, 60, 4
    tgt = rng.standard_normal((B * (D + 1), V)).astype(np.float32)
    drf = np.empty((B * D, V), dtype=np.float32)
    toks = np.empty(B * D, dtype=np.int32)
    for b in range(B):
        for j in range(D):
            r = tgt[b * (D + 1) + j]
            if j == 2:
                r[j] = -np.inf               # token j: probability 0 in both rows
            drf[b * D + j] = r
            toks[b * D + j] = j if j == 2 else int(np.argmax(r))
    ua = rng.random(B * D, dtype=np.float32) * np.float32(0.99)
    us = rng.random(B, dtype=np.float32)
    al, nt, _, _ = oracle.accept_stochastic(tgt, drf, toks, np.full(B, D, np.int32), ua, us)
    assert np.all(al == 3)
    for b in range(B):
        p2 = _softmax(tgt[b * (D + 1) + 2].astype(np.float64))
        assert nt[b] == _inverse_cdf(p2, float(us[b])) and nt[b] != 2


def test_decision_margins_closed_forms():
    """Signed decision margins, (p(x) - u q(x)) / max(p(x), u q(x)):
    * q = p: 1 - u at every position (kept unless u = 1);
    * a drafter certain of x where p(x) = 0: -1 (rejected), or 0 when u = 0;
    * two-token rows p = (a, 1 - a), q = (b, 1 - b), x = 0: (a - u b) / max(a, u b).
    And the acceptance length is 1 + the number of leading positive decisions."""
    rng = np.random.default_rng(23)
    B, D, V = 20, 5, 40
    tgt = rng.standard_normal((B * (D + 1), V)).astype(np.float32)
    drf = np.concatenate([tgt[b * (D + 1):b * (D + 1) + D] for b in range(B)])
    toks = rng.integers(0, V, size=B * D).astype(np.int32)
    ua = rng.random(B * D, dtype=np.float32)
    dm = oracle.stochastic_decisions(tgt, drf, toks, np.full(B, D, np.int32), ua)
    assert np.allclose(dm, 1.0 - ua.astype(np.float64), rtol=0, atol=1e-12)

    tg = rng.standard_normal((2 * 8, V)).astype(np.float32)
    dr = np.full((8, V), -1e30, dtype=np.float32)
    x = rng.integers(0, V, size=8).astype(np.int32)
    for b in range(8):
        tg[2 * b, x[b]] = -np.inf
        dr[b, x[b]] = 0.0
    u = rng.random(8, dtype=np.float32)
    u[0] = 0.0
    dm = oracle.stochastic_decisions(tg, dr, x, np.ones(8, np.int32), u)
    assert dm[0] == 0.0 and np.all(dm[1:] == -1.0)

    a = rng.uniform(0.05, 0.95, size=30)
    b = rng.uniform(0.05, 0.95, size=30)
    u = rng.random(30, dtype=np.float32)
    lt = np.log(np.stack([a, 1 - a], axis=1))
    ld = np.log(np.stack([b, 1 - b], axis=1))
    tgt2 = np.repeat(lt, 2, axis=0).astype(np.float32)   # rows 0 and 1 of each sequence
    drf2 = ld.astype(np.float32)
    dm = oracle.stochastic_decisions(tgt2, drf2, np.zeros(30, np.int32), np.ones(30, np.int32), u)
    pa = _softmax_rows(lt.astype(np.float32).astype(np.float64))[:, 0]
    qb = _softmax_rows(ld.astype(np.float32).astype(np.float64))[:, 0]
    lhs, rhs = u.astype(np.float64) * qb, pa
    assert np.allclose(dm, (rhs - lhs) / np.maximum(lhs, rhs), rtol=1e-12, atol=1e-15)

    # the acceptance path follows the signs
    drf3 = (tgt[[b * (D + 1) + j for b in range(B) for j in range(D)]]
            + rng.standard_normal((B * D, V)).astype(np.float32) * 0.5)
    toks3 = np.array([int(np.argmax(r)) for r in drf3], dtype=np.int32)
    al, _, _, _ = oracle.accept_stochastic(tgt, drf3, toks3, np.full(B, D, np.int32), ua,
                                           rng.random(B, dtype=np.float32))
    dm = oracle.stochastic_decisions(tgt, drf3, toks3, np.full(B, D, np.int32), ua).reshape(B, D)
    lead = np.array([int(np.argmin(np.append(r > 0, False))) for r in dm])
    assert np.array_equal(al, lead + 1)
    assert 0 < (al - 1).mean() < D


def _softmax_rows(x):
    z = np.exp(x - x.max(axis=1, keepdims=True))
    return z / z.sum(axis=1, keepdims=True)
