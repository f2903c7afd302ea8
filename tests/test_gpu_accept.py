"""GPU parity of spec_accept against the oracle: bit-exact target tokens, acceptance
lengths and next tokens, on every workload at full size and on edge cases."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_gqa_gb300 import synth

from gpu_util import dev_accept, ensure_built, gpu_accept

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _check(a, max_draft=None):
    al, nt, tgt = gpu_accept(a, max_draft)
    ral, rnt, ramax = oracle.spec_accept(a["logits"], a["draft_tokens"], a["draft_len"])
    assert np.array_equal(tgt, ramax)
    assert np.array_equal(al, ral)
    assert np.array_equal(nt, rnt)
    assert np.all(al >= 1) and np.all(al <= a["draft_len"] + 1)
    return al


@pytest.mark.parametrize("cfg", ["c1", "c2", "c3", "c4", "c5"])
def test_full_size_workloads(cfg):
    w = synth.CONFIGS[cfg]
    a = synth.accept_inputs(w, 1)
    al = _check(a)
    if cfg != "c1":
        assert al.max() > 1  # drafts do get accepted


@pytest.mark.parametrize("D", synth.C4_SWEEP_D)
def test_tile_sweep_draft_lengths(D):
    w = synth.CONFIGS["c4"].with_(B=8)
    T, Dv, p = synth.lengths(w, 2, D=D)
    _check(synth.accept_inputs(w, 2, draft_len=Dv, p=p))


@pytest.mark.parametrize("V,dtype", [(1, "bf16"), (7, "fp32"), (13, "bf16"), (1001, "bf16"),
                                     (1001, "fp32"), (32003, "bf16"), (65537, "fp32")])
def test_ragged_vocab_and_alignment(V, dtype):
    """V not a multiple of the vector width: rows start at unaligned addresses."""
    w = synth.Workload("v", B=5, Hq=1, Hkv=1, d=8, D=3, T=1, V=V, p=0.8, logits_dtype=dtype)
    Dv = np.array([3, 0, 1, 3, 2], dtype=np.int32)
    _check(synth.accept_inputs(w, 3, draft_len=Dv, p=np.full(5, 0.8)), max_draft=4)


def test_ties_and_signed_zero():
    V = 4099
    rows = 4
    logits = np.full((rows, V), -1.0, dtype=np.float32)
    logits[0, [5, 4000, 4098]] = 3.0
    logits[1, :] = 0.0
    logits[1, 2:7] = -0.0
    logits[2, [17, 4097]] = 2.0
    logits[3, 4098] = 9.0
    for dt in ("fp32", "bf16"):
        lg = logits if dt == "fp32" else synth.bf16_bits(logits)
        a = dict(logits=lg, draft_tokens=np.array([5, 0, 17], dtype=np.int32),
                 draft_len=np.array([3], dtype=np.int32))
        al, nt, tgt = gpu_accept(a)
        assert list(tgt) == [5, 0, 17, 4098]
        assert al[0] == 4 and nt[0] == 4098


def test_reuse_workspace_and_repeat():
    import speculative_decoding_verification_gqa_gb300 as sv
    w = synth.CONFIGS["c2"].with_(B=4)
    a = synth.accept_inputs(w, 4)
    lg, dt, dl = dev_accept(a)
    ws = sv.new_workspace(sv.accept_workspace_bytes(4, 31, w.V))
    r1 = [t.cpu().clone() for t in sv.spec_accept(lg, dt, dl, max_draft_len=31, workspace=ws)]
    r2 = [t.cpu().clone() for t in sv.spec_accept(lg, dt, dl, max_draft_len=31, workspace=ws)]
    assert all(torch.equal(x, y) for x, y in zip(r1, r2))
    assert sv.workspace_status(ws) == 0


def test_device_side_length_check_sets_flag():
    import speculative_decoding_verification_gqa_gb300 as sv
    w = synth.Workload("e", B=3, Hq=1, Hkv=1, d=8, D=2, T=1, V=64, p=0.5, logits_dtype="fp32")
    a = synth.accept_inputs(w, 5)
    lg, dt, dl = dev_accept(a)
    ws = sv.new_workspace(sv.accept_workspace_bytes(3, 1, 64))
    al = torch.full((3,), -7, dtype=torch.int32, device="cuda")
    nt = torch.full((3,), -7, dtype=torch.int32, device="cuda")
    sv.spec_accept(lg, dt, dl, max_draft_len=1, accept_len=al, next_token=nt, workspace=ws)
    assert sv.workspace_status(ws, clear=True) == 8
    assert (al.cpu() == -7).all() and (nt.cpu() == -7).all()
    assert sv.workspace_status(ws) == 0


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_subnormal_and_nan_values(dtype):
    """A positive subnormal is the maximum of a row of zeros and negatives (the packed
    vector maximum must not flush it); NaN never wins, and later equal values lose."""
    V = 1037
    rows = 4
    logits = np.full((rows, V), -2.0, dtype=np.float32)
    tiny = np.array([0x0001 if dtype == "bf16" else 0x00000001], dtype=np.uint32)
    tiny = (tiny << 16).view(np.float32)[0] if dtype == "bf16" else tiny.view(np.float32)[0]
    logits[0, :] = 0.0
    logits[0, 700] = tiny
    logits[0, 900] = tiny
    logits[1, [3, 17, 500]] = np.nan
    logits[1, 400] = 5.0
    logits[1, 401] = 5.0
    logits[2, :] = -np.inf
    logits[2, 1036] = -1.0
    logits[3, :] = -np.inf
    logits[3, 0] = np.nan
    lg = logits if dtype == "fp32" else synth.bf16_bits(logits)
    a = dict(logits=lg, draft_tokens=np.array([700, 400, 1036], dtype=np.int32),
             draft_len=np.array([3], dtype=np.int32))
    al, nt, tgt = gpu_accept(a)
    assert list(tgt) == [700, 400, 1036, 1]
    assert al[0] == 4 and nt[0] == 1


def test_workspace_shared_by_shapes_and_after_a_failed_check():
    """One workspace, sized for the largest call, serves calls of different shapes (and so
    different CTA counts) back to back, including after a call whose device-side length
    check failed."""
    import speculative_decoding_verification_gqa_gb300 as sv
    ws = sv.new_workspace(sv.accept_workspace_bytes(8, 15, 128256))
    for B, V, md in [(8, 128256, 15), (3, 1000, 4), (8, 32000, 15), (1, 64, 2)]:
        w = synth.Workload("w", B=B, Hq=1, Hkv=1, d=8, D=md, T=1, V=V, p=0.7)
        a = synth.accept_inputs(w, B + V)
        lg, dt, dl = dev_accept(a)
        if B == 3:  # D_0 > max_draft_len: the call fails on the device
            bad = dl.clone()
            bad[0] = md + 1
            sv.spec_accept(lg, dt, bad, max_draft_len=md, workspace=ws)
            assert sv.workspace_status(ws, clear=True) == 8
        al, nt = sv.spec_accept(lg, dt, dl, max_draft_len=md, workspace=ws)
        torch.cuda.synchronize()
        assert sv.workspace_status(ws) == 0
        ral, rnt, _ = oracle.spec_accept(a["logits"], a["draft_tokens"], a["draft_len"])
        assert np.array_equal(al.cpu().numpy(), ral) and np.array_equal(nt.cpu().numpy(), rnt)


@pytest.mark.parametrize("B,D,V", [(300, 15, 64), (1100, 3, 16)])
def test_many_rows_and_sequences(B, D, V):
    """More window rows (4800, 4400) than the last CTA keeps in shared memory, and more
    sequences (1100) than it keeps draft lengths for: the global-memory fallback."""
    w = synth.Workload("m", B=B, Hq=1, Hkv=1, d=8, D=D, T=1, V=V, p=0.8)
    _check(synth.accept_inputs(w, 9))


@pytest.mark.parametrize("V,dtype", [(1072, "bf16"), (536, "fp32"), (16, "bf16")])
def test_row_boundaries_inside_a_batch(V, dtype):
    """Rows of whole 32-byte vectors, 67 per row (coprime with the CTAs' batches) or one:
    the continuous scan meets row ends at every offset of a batch and of a CTA's range.
    Row kinds cycle so that a vector counted in the wrong row changes a result: 5 at the
    last element; 6 at the first and the last (tie: the first); all -1 (tie: the first).
    The argmax of each row is known in closed form; acceptance is checked by the oracle."""
    B, D = 200, 4
    R = B * (D + 1)
    kind = np.arange(R) % 3
    x = np.zeros((R, V), dtype=np.float32)
    x[kind == 0, V - 1] = 5.0
    x[kind == 1, 0] = 6.0
    x[kind == 1, V - 1] = 6.0
    x[kind == 2, :] = -1.0
    expect = np.where(kind == 0, V - 1, 0).astype(np.int32)
    logits = synth.bf16_bits(x) if dtype == "bf16" else x
    draft_len = np.full(B, D, dtype=np.int32)
    drafts = []
    for b in range(B):
        t = expect[b * (D + 1):b * (D + 1) + D].copy()
        if b % 5 < D:
            t[b % 5] = (t[b % 5] + 1) % V  # first mismatch at position b % 5
        drafts.append(t)
    a = {"logits": logits, "draft_tokens": np.concatenate(drafts).astype(np.int32),
         "draft_len": draft_len}
    al, nt, tgt = gpu_accept(a, D)
    assert np.array_equal(tgt, expect)
    ral, rnt, ramax = oracle.spec_accept(a["logits"], a["draft_tokens"], a["draft_len"])
    assert np.array_equal(ramax, expect)
    assert np.array_equal(al, ral) and np.array_equal(nt, rnt)
    assert np.array_equal(al, np.minimum(np.arange(B) % 5, D) + 1)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_aligned_and_unaligned_logits(dtype):
    """The same logits on 16-byte row boundaries and shifted by one element (every row then
    has a scalar head and tail around its 16-byte vectors): both match the oracle."""
    import speculative_decoding_verification_gqa_gb300 as sv
    w = synth.Workload("a", B=6, Hq=1, Hkv=1, d=8, D=7, T=1, V=4096, p=0.75, logits_dtype=dtype)
    a = synth.accept_inputs(w, 21)
    lg, dt, dl = dev_accept(a)
    flat = torch.empty(lg.numel() + 8, dtype=lg.dtype, device="cuda")
    shifted = flat[1:1 + lg.numel()].view(lg.shape)
    shifted.copy_(lg)
    ral, rnt, ramax = oracle.spec_accept(a["logits"], a["draft_tokens"], a["draft_len"])
    for x in (lg, shifted):
        tgt = torch.full((lg.shape[0],), -1, dtype=torch.int32, device="cuda")
        al, nt = sv.spec_accept(x, dt, dl, max_draft_len=7, target_tokens=tgt)
        torch.cuda.synchronize()
        assert np.array_equal(tgt.cpu().numpy(), ramax)
        assert np.array_equal(al.cpu().numpy(), ral) and np.array_equal(nt.cpu().numpy(), rnt)


@pytest.mark.parametrize("B,D,V", [(16, 31, 128256), (300, 15, 64), (5, 0, 1000), (1, 255, 300)])
def test_every_call_leaves_the_workspace_at_zero(B, D, V):
    """The last CTA clears the row keys, the completion ticket and any target-token
    scratch, so a zero-filled workspace is zero again after every call (here including
    sequences spread over many CTAs, more rows than the last CTA keeps in shared memory,
    no drafts at all, and the longest window)."""
    import speculative_decoding_verification_gqa_gb300 as sv
    w = synth.Workload("z", B=B, Hq=1, Hkv=1, d=8, D=D, T=1, V=V, p=0.9)
    a = synth.accept_inputs(w, 31)
    lg, dt, dl = dev_accept(a)
    ws = sv.new_workspace(sv.accept_workspace_bytes(B, D, V))
    for _ in range(2):
        al, nt = sv.spec_accept(lg, dt, dl, max_draft_len=D, workspace=ws)
        torch.cuda.synchronize()
        assert int(torch.count_nonzero(ws)) == 0
        ral, rnt, _ = oracle.spec_accept(a["logits"], a["draft_tokens"], a["draft_len"])
        assert np.array_equal(al.cpu().numpy(), ral) and np.array_equal(nt.cpu().numpy(), rnt)
