"""GPU parity of spec_accept_stochastic against the fp64 oracle.

Where floating point decides an integer here, fp32 and fp64 may legitimately differ:
* a keep / reject decision u q(x) < p(x) whose two sides are closer than ACC_MARGIN
  (relative) may go either way: p(x) and q(x) carry relative errors of about 1e-6 in
  fp32;
* a draw picks the token whose interval of the running sum holds u times the total; the
  fp32 running sums over up to 128K weights (per-thread segments, a scan of 256 segment
  sums in each of the 8 CTAs that share the row, then the 8 CTA totals) are within
  CDF_TOL of the total, so near an interval's end a neighbour may be drawn. For a flat softmax over a large vocabulary the intervals are themselves
  about 1e-5 of the total.
So every keep / reject decision on the GPU's path must agree with the oracle's wherever
the oracle's margin for that decision is at least ACC_MARGIN: the GPU may leave the
oracle's path only at a position whose own margin is below it (every decision is checked,
also on sequences with a low-margin decision elsewhere). Where the two paths agree, the
token must equal the oracle's where the draw's margin is at least CDF_TOL; elsewhere, and
on a path that left the oracle's at a low-margin position, it must be a valid draw from
the GPU path's weights: a token of positive weight whose fp64 interval lies within CDF_TOL
of u times the total. Nothing else differs."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_gqa_gb300 as sv
from speculative_decoding_verification_gqa_gb300 import synth

from gpu_util import ensure_built

pytestmark = pytest.mark.gpu

ACC_MARGIN = 1e-4
CDF_TOL = 3e-5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _dev_logits(a):
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(a).cuda()


def _f64(a):
    return ((a.astype(np.uint32) << np.uint32(16)).view(np.float32)
            if a.dtype == np.uint16 else a).astype(np.float64)


def gpu_stochastic(x, temperature, max_draft=None, ws=None, outs=None):
    md = int(x["draft_len"].max()) if max_draft is None else max_draft
    al, nt = sv.spec_accept_stochastic(
        _dev_logits(x["target_logits"]), _dev_logits(x["draft_logits"]),
        torch.from_numpy(x["draft_tokens"]).cuda(), torch.from_numpy(x["draft_len"]).cuda(),
        torch.from_numpy(x["u_accept"]).cuda(), torch.from_numpy(x["u_sample"]).cuda(),
        max_draft_len=md, temperature=temperature, workspace=ws,
        accept_len=None if outs is None else outs[0], next_token=None if outs is None else outs[1])
    torch.cuda.synchronize()
    return al.cpu().numpy(), nt.cpu().numpy()


def _draw_weights(x, b, n, temperature):
    """fp64 weights of sequence b's draw after n kept drafts (max(0, p - q), or p)."""
    D = x["draft_len"]
    q_off = int(np.sum(D[:b] + 1))
    d_off = int(np.sum(D[:b]))
    sm = lambda r: (lambda z: z / z.sum())(np.exp((r / temperature) - (r / temperature).max()))
    p = sm(_f64(x["target_logits"][q_off + n]))
    if n < D[b]:
        w = np.maximum(p - sm(_f64(x["draft_logits"][d_off + n])), 0.0)
        return w if w.sum() > 0 else p
    return p


def _valid_draw(x, b, n, temperature, tok):
    w = _draw_weights(x, b, n, temperature)
    c = np.cumsum(w)
    t = float(x["u_sample"][b]) * c[-1]
    lo = c[tok - 1] if tok > 0 else 0.0
    return w[tok] > 0 and lo - CDF_TOL * c[-1] <= t <= c[tok] + CDF_TOL * c[-1]


def check(x, temperature, min_decided=0.5):
    al, nt = gpu_stochastic(x, temperature)
    ral, rnt, ma, ms = oracle.accept_stochastic(
        x["target_logits"], x["draft_logits"], x["draft_tokens"], x["draft_len"],
        x["u_accept"], x["u_sample"], temperature)
    dm = oracle.stochastic_decisions(x["target_logits"], x["draft_logits"], x["draft_tokens"],
                                     x["draft_len"], x["u_accept"], temperature)
    D = x["draft_len"]
    d_off = np.concatenate([[0], np.cumsum(D.astype(np.int64))])
    assert np.all((al >= 1) & (al <= D + 1))
    raw_diff = 0
    for b in range(len(D)):
        n = int(al[b]) - 1            # drafts the GPU kept
        sb = dm[d_off[b]:d_off[b + 1]]
        firm = np.abs(sb) >= ACC_MARGIN
        # kept on the GPU: positions 0..n-1; rejected: position n (if n < D)
        assert not np.any(firm[:n] & (sb[:n] <= 0)), (b, n, sb[:n + 1])
        if n < D[b]:
            assert not (firm[n] and sb[n] > 0), (b, n, sb[n])
        raw_diff += int(al[b] != ral[b])
    decided = ma >= ACC_MARGIN
    assert np.array_equal(al[decided], ral[decided]), (al, ral, ma)
    assert decided.mean() >= min_decided
    for b in range(len(D)):
        if al[b] == ral[b] and ms[b] >= CDF_TOL:
            assert nt[b] == rnt[b], (b, nt[b], rnt[b], ms[b])
        else:
            assert _valid_draw(x, b, int(al[b]) - 1, temperature, int(nt[b])), (b, nt[b])
    print("sequences %d, acceptance lengths differing at a low-margin decision: %d"
          % (len(D), raw_diff))
    return al, nt


# V = 7 and 32003: rows off 16-byte boundaries (scalar loads); 1000 and 128256: one batch of
# 16-byte loads per thread and row slice (the next position's loads overlap this one's
# reductions); 262144: several batches per slice
CASES = [(7, "fp32", 1.0), (7, "bf16", 0.3), (1000, "bf16", 1.0), (1000, "fp32", 0.3),
         (32003, "bf16", 0.3), (32003, "fp32", 1.0), (128256, "bf16", 0.3),
         (262144, "bf16", 1.0)]


@pytest.mark.parametrize("V,dtype,temperature", CASES)
def test_ragged_batches(V, dtype, temperature):
    w = synth.Workload("s", B=12, Hq=1, Hkv=1, d=8, D=7, T=1, V=V, p=0.8, logits_dtype=dtype)
    Dv = np.array([7, 0, 3, 7, 1, 5, 2, 7, 0, 4, 6, 7], dtype=np.int32)
    x = synth.stochastic_inputs(w, V % 97, draft_len=Dv, noise=0.2)
    check(x, temperature)


@pytest.mark.parametrize("temperature", [0.3, 1.0])
def test_full_size_llama3_8b_shape(temperature):
    """16 sequences of 31 drafts over a 128,256-token vocabulary, bf16 logits."""
    w = synth.CONFIGS["c2"]
    x = synth.stochastic_inputs(w, 1, noise=0.1)
    al, _ = check(x, temperature, min_decided=0.8)
    if temperature == 0.3:
        assert al.max() > 1


def test_drafter_equal_to_target_keeps_every_draft():
    w = synth.Workload("e", B=8, Hq=1, Hkv=1, d=8, D=6, T=1, V=5000, p=0.5)
    x = synth.stochastic_inputs(w, 2)
    D = x["draft_len"]
    rows = [int(np.sum(D[:b] + 1)) + j for b in range(len(D)) for j in range(int(D[b]))]
    x["draft_logits"] = x["target_logits"][rows].copy()
    al, _ = check(x, 1.0, min_decided=1.0)
    assert np.array_equal(al, D + 1)


def test_one_token_vocabulary():
    w = synth.Workload("v1", B=4, Hq=1, Hkv=1, d=8, D=3, T=1, V=1, p=0.5, logits_dtype="fp32")
    x = synth.stochastic_inputs(w, 4)
    al, nt = gpu_stochastic(x, 1.0)
    assert np.array_equal(al, x["draft_len"] + 1) and np.all(nt == 0)


def test_repeatable_and_device_checks():
    w = synth.Workload("r", B=5, Hq=1, Hkv=1, d=8, D=4, T=1, V=3000, p=0.8)
    x = synth.stochastic_inputs(w, 6)  # every D_b = 4
    ws = sv.new_workspace(256)
    a1 = gpu_stochastic(x, 0.5, ws=ws)
    a2 = gpu_stochastic(x, 0.5, ws=ws)
    assert all(np.array_equal(p, q) for p, q in zip(a1, a2))
    assert sv.workspace_status(ws) == 0

    def fresh():
        return (torch.full((5,), -7, dtype=torch.int32, device="cuda"),
                torch.full((5,), -7, dtype=torch.int32, device="cuda"))

    # D_0 = 5 above max_draft_len = 4: every sequence's offsets depend on it, so every
    # sequence is left untouched
    bad = dict(x, draft_len=x["draft_len"].copy())
    bad["draft_len"][0] = 5
    outs = fresh()
    gpu_stochastic(bad, 0.5, max_draft=4, ws=ws, outs=outs)
    assert sv.workspace_status(ws, clear=True) == 8
    assert (outs[0] == -7).all() and (outs[1] == -7).all()
    # a draft token outside the vocabulary: that sequence alone is left untouched
    tok = dict(x, draft_tokens=x["draft_tokens"].copy())
    tok["draft_tokens"][0] = 3000
    outs = fresh()
    gpu_stochastic(tok, 0.5, ws=ws, outs=outs)
    assert sv.workspace_status(ws, clear=True) == 8
    assert int(outs[0][0]) == -7 and int(outs[1][0]) == -7
    assert bool((outs[0][1:] != -7).all()) and bool((outs[1][1:] != -7).all())


def test_all_zero_residual_draws_from_the_target():
    """p = q at a draft position and the drafted token impossible under both (logit -inf in
    both rows): the draft is rejected (0 < 0 fails) and every weight of max(0, p - q) is 0,
    so the token is drawn from the target's row of that position."""
    V = 5000
    w = synth.Workload("z", B=6, Hq=1, Hkv=1, d=8, D=3, T=1, V=V, p=0.5, logits_dtype="fp32")
    x = synth.stochastic_inputs(w, 8, noise=0.2)
    D = x["draft_len"]
    rng = np.random.default_rng(9)
    d_off = 0
    for b in range(len(D)):
        q_off = d_off + b
        if D[b] >= 1:
            j = int(rng.integers(D[b]))
            tok = int(rng.integers(V))
            row = x["target_logits"][q_off + j].copy()
            row[tok] = -np.inf
            x["target_logits"][q_off + j] = row
            x["draft_logits"][d_off + j] = row
            x["draft_tokens"][d_off + j] = tok
            # the drafts before it are the drafter's copies of the target (kept for u < 1)
            for jj in range(j):
                x["draft_logits"][d_off + jj] = x["target_logits"][q_off + jj]
        d_off += int(D[b])
    al, nt = check(x, 1.0, min_decided=0.0)
    ral, _, _, _ = oracle.accept_stochastic(
        x["target_logits"], x["draft_logits"], x["draft_tokens"], x["draft_len"],
        x["u_accept"], x["u_sample"], 1.0)
    assert np.array_equal(al, ral)
