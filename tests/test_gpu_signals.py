"""GPU parity of spec_draft_signals against the fp64 oracle (largest softmax probability
and entropy per row).

Tolerance: the kernel works in fp32 with ex2.approx (measured relative error up to about
2^-19 per element, e.g. at 0) and sums up to V terms per row through per-thread, warp and CTA partials, so the
row sum z carries a relative error of order 1e-6; confidence = 1/z inherits it, and
entropy = ln z - ln2 * s / z (s/z up to log2 V, about 17) an absolute error of order
1e-5. The bounds below are 2e-5 relative on the confidence and 1e-4 absolute (nats) on the
entropy."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_gqa_gb300 as sv
from speculative_decoding_verification_gqa_gb300 import synth

from gpu_util import ensure_built

pytestmark = pytest.mark.gpu

CONF_RTOL = 2e-5
ENT_ATOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _dev(logits):
    if logits.dtype == np.uint16:
        return torch.from_numpy(logits.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(logits).cuda()


def _check(logits, ws=None):
    conf, ent = sv.spec_draft_signals(_dev(logits), workspace=ws)
    torch.cuda.synchronize()
    rc, re = oracle.draft_signals(logits)
    c = conf.cpu().numpy().astype(np.float64)
    e = ent.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(c - rc) <= CONF_RTOL * rc), np.max(np.abs(c - rc) / rc)
    assert np.all(np.abs(e - re) <= ENT_ATOL), np.max(np.abs(e - re))
    return c, e


def _rows(rows, V, seed, dtype):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, V)) * rng.choice([0.1, 1.0, 3.0, 8.0], size=(rows, 1))
    x = x.astype(np.float32)
    return synth.bf16_bits(x) if dtype == "bf16" else x


@pytest.mark.parametrize("rows,V,dtype", [(4, 1000, "fp32"), (7, 32000, "bf16"),
                                          (3, 128256, "bf16"), (5, 1001, "fp32"),
                                          (9, 1001, "bf16"), (64, 7, "bf16"), (2, 65537, "fp32"),
                                          # rows of 67 and 97 32-byte vectors: row ends at every
                                          # offset of a batch (the continuous path)
                                          (200, 1072, "bf16"), (300, 776, "fp32"),
                                          # about 14 rows per CTA range: near its limit
                                          (1000, 640, "bf16"),
                                          # more rows per range than it takes: row by row
                                          (5000, 16, "bf16")])
def test_random_rows(rows, V, dtype):
    """Confidence and entropy of seeded rows against the oracle, across both scans: the
    continuous one (rows of whole 32-byte vectors, at most 16 rows per CTA range) and the
    row-by-row one (any other shape)."""
    _check(_rows(rows, V, rows * 1000 + V, dtype))


def test_closed_forms_and_special_rows():
    """Uniform row (1/V, ln V); one dominant logit (about 1, about 0); two equal maxima
    with the rest at -inf (1/2, ln 2); -inf and NaN mixed into a random row; V = 1."""
    V = 4099
    x = np.random.default_rng(3).standard_normal((5, V)).astype(np.float32)
    x[0, :] = 0.5
    x[1, 17] = 60.0
    x[2, :] = -np.inf
    x[2, [5, 4000]] = 1.25
    x[3, ::3] = -np.inf
    c, e = _check(x[:4])
    assert c[0] == pytest.approx(1.0 / V, rel=CONF_RTOL) and e[0] == pytest.approx(np.log(V), abs=ENT_ATOL)
    assert c[1] == pytest.approx(1.0, rel=CONF_RTOL) and e[1] == pytest.approx(0.0, abs=ENT_ATOL)
    assert c[2] == pytest.approx(0.5, rel=CONF_RTOL) and e[2] == pytest.approx(np.log(2.0), abs=ENT_ATOL)
    one = np.array([[2.5]], dtype=np.float32)
    c1, e1 = _check(one)
    assert c1[0] == pytest.approx(1.0, rel=CONF_RTOL) and abs(e1[0]) <= ENT_ATOL
    # NaN elements are ignored
    y = x[4:5].copy()
    ref_c, ref_e = oracle.draft_signals(y)
    y[0, [3, 100, 4098]] = np.nan
    conf, ent = sv.spec_draft_signals(_dev(y))
    keep = np.ones(V, bool)
    keep[[3, 100, 4098]] = False
    rc, re = oracle.draft_signals(np.ascontiguousarray(x[4:5, keep]))
    assert abs(conf.item() - rc[0]) <= CONF_RTOL * rc[0] and abs(ent.item() - re[0]) <= ENT_ATOL


def test_full_size_logits_of_the_llama3_8b_step():
    """The c2-shaped matrix: 512 rows of 128,256 bf16 logits, every row checked."""
    w = synth.CONFIGS["c2"]
    a = synth.accept_inputs(w, 1)
    _check(a["logits"])


def test_workspace_shared_by_shapes():
    """One workspace serves calls of different shapes (and so CTA counts) back to back."""
    ws = sv.new_workspace(sv.signals_workspace_bytes(512, 128256))
    for rows, V, dt in [(512, 128256, "bf16"), (3, 999, "fp32"), (40, 32000, "bf16"), (1, 8, "fp32")]:
        _check(_rows(rows, V, 7 + rows, dt), ws=ws)
