"""Failure paths on the GPU, made on the host. A launch failure injected at each kernel
launch of every call (sv_inject_launch_failure) is reported as SV_ERR_CUDA, leaves what
the call must not touch untouched, and the next call on the same workspace is correct
again. Guard bands around every output buffer stay unchanged by ordinary calls. Nothing
here faults, traps or hangs the GPU."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_gqa_gb300 as sv
from speculative_decoding_verification_gqa_gb300 import synth

from gpu_util import assert_close, dev_accept, dev_attn, ensure_built, oracle_attn

pytestmark = pytest.mark.gpu

SENT = 7.0


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()
    yield
    sv.api.inject_launch_failure(-1)


def _attn_case():
    w = synth.Workload("f", B=3, Hq=16, Hkv=4, d=128, D=0, T=0, V=8, p=0.5)
    x = synth.attn_inputs(w, 17, seq_lens=np.array([900, 5, 300]), draft_len=np.array([7, 0, 3]))
    return w, x


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("after", [0, 1, 2])
@pytest.mark.parametrize("entry", ["packed", "host_lengths"])
def test_verify_attn_reports_a_failed_launch_and_recovers(after, entry):
    w, x = _attn_case()
    q, k, v, sc, T, D = dev_attn(x)
    Th = torch.from_numpy(x["seq_lens"].astype(np.int32))
    Dh = torch.from_numpy(x["draft_len"].astype(np.int32))
    ws = sv.new_workspace(sv.verify_workspace_bytes(sv.api.attn_desc(q, k, 3, 7, 900)))
    out = torch.full_like(q, SENT)

    def call():
        if entry == "packed":
            return sv.spec_verify_attn(q, k, v, T, D, max_draft_len=7, max_seq_len=900,
                                       out=out, workspace=ws)
        return sv.spec_verify_attn_host_lengths(q, k, v, T, D, Th, Dh, max_draft_len=7,
                                                max_seq_len=900, out=out, workspace=ws)

    launches = 3 if entry == "packed" else 2
    sv.api.inject_launch_failure(after)
    if after < launches:
        with pytest.raises(sv.SpecVerifyError) as e:
            call()
        assert e.value.status == 6
        assert sv.api.inject_launch_failure(-1) == -1  # the failure was used
        torch.cuda.synchronize()
        if after < launches - 1:  # the attention kernel never ran: out untouched
            assert (out == SENT).all()
    else:  # armed beyond this call: the call succeeds and the failure stays pending
        call()
        assert sv.api.inject_launch_failure(-1) == after - launches
    call()
    torch.cuda.synchronize()
    assert sv.workspace_status(ws) == 0
    assert_close(_bits(out), oracle_attn(w, x))


@pytest.mark.parametrize("which", ["accept", "signals"])
def test_logits_calls_report_a_failed_launch_and_recover(which):
    wk = synth.Workload("f", B=4, Hq=1, Hkv=1, d=8, D=5, T=1, V=5000, p=0.8)
    a = synth.accept_inputs(wk, 23)
    lg, dt, dl = dev_accept(a)
    if which == "accept":
        ws = sv.new_workspace(sv.accept_workspace_bytes(4, 5, 5000))
        al = torch.full((4,), -7, dtype=torch.int32, device="cuda")
        nt = torch.full((4,), -7, dtype=torch.int32, device="cuda")
        call = lambda: sv.spec_accept(lg, dt, dl, max_draft_len=5, accept_len=al,
                                      next_token=nt, workspace=ws)
        outs = (al, nt)
    else:
        ws = sv.new_workspace(sv.signals_workspace_bytes(lg.shape[0], 5000))
        cf = torch.full((lg.shape[0],), SENT, device="cuda")
        en = torch.full((lg.shape[0],), SENT, device="cuda")
        call = lambda: sv.spec_draft_signals(lg, confidence=cf, entropy=en, workspace=ws)
        outs = (cf, en)
    sv.api.inject_launch_failure(0)
    with pytest.raises(sv.SpecVerifyError) as e:
        call()
    assert e.value.status == 6
    torch.cuda.synchronize()
    assert all(bool((o == (-7 if o.dtype == torch.int32 else SENT)).all()) for o in outs)
    call()
    torch.cuda.synchronize()
    assert sv.workspace_status(ws) == 0
    if which == "accept":
        ral, rnt, _ = oracle.spec_accept(a["logits"], a["draft_tokens"], a["draft_len"])
        assert np.array_equal(al.cpu().numpy(), ral) and np.array_equal(nt.cpu().numpy(), rnt)
        assert int(torch.count_nonzero(ws)) == 0
    else:
        rc, re = oracle.draft_signals(a["logits"])  # the signals tests' bounds
        assert np.all(np.abs(cf.cpu().numpy().astype(np.float64) - rc) <= 2e-5 * rc)
        assert np.all(np.abs(en.cpu().numpy().astype(np.float64) - re) <= 1e-4)


def _guarded(n, dtype, fill, pad=64):
    """A view of n elements inside a buffer with `pad` guard elements on each side (the
    view keeps 16-byte alignment)."""
    buf = torch.full((n + 2 * pad,), fill, dtype=dtype, device="cuda")
    return buf, buf[pad:pad + n]


def _guards_intact(buf, n, fill, pad=64):
    return bool((buf[:pad] == fill).all()) and bool((buf[pad + n:] == fill).all())


@pytest.mark.parametrize("kernel", [1, 2], ids=["mma", "tcgen05"])
@pytest.mark.parametrize("window", [0, 100])
def test_attention_writes_nothing_outside_out(kernel, window):
    w, x = _attn_case()
    q, k, v, sc, T, D = dev_attn(x)
    prev = sv.set_attn_kernel(kernel)
    try:
        n = q.numel()
        pad = 16 * 128  # whole rows of Hq x d on each side
        buf, flat = _guarded(n, torch.bfloat16, SENT, pad)
        out = flat.view(q.shape)
        sv.spec_verify_attn(q, k, v, T, D, max_draft_len=7, max_seq_len=900, out=out,
                            sliding_window=window)
        torch.cuda.synchronize()
        assert _guards_intact(buf, n, SENT, pad)
        assert_close(_bits(out), oracle_attn(w, x, window=window))
    finally:
        sv.set_attn_kernel(prev)


def test_accept_and_signals_write_nothing_outside_their_outputs():
    wk = synth.Workload("g", B=6, Hq=1, Hkv=1, d=8, D=4, T=1, V=3001, p=0.8)
    a = synth.accept_inputs(wk, 29)
    lg, dt, dl = dev_accept(a)
    rows = lg.shape[0]
    ab, al = _guarded(6, torch.int32, -7)
    nb, nt = _guarded(6, torch.int32, -7)
    tb, tg = _guarded(rows, torch.int32, -7)
    sv.spec_accept(lg, dt, dl, max_draft_len=4, accept_len=al, next_token=nt, target_tokens=tg)
    cb, cf = _guarded(rows, torch.float32, SENT)
    eb, en = _guarded(rows, torch.float32, SENT)
    sv.spec_draft_signals(lg, confidence=cf, entropy=en)
    torch.cuda.synchronize()
    for b_, n_ in ((ab, 6), (nb, 6), (tb, rows)):
        assert _guards_intact(b_, n_, -7)
    for b_ in (cb, eb):
        assert _guards_intact(b_, rows, SENT)
    ral, rnt, ramax = oracle.spec_accept(a["logits"], a["draft_tokens"], a["draft_len"])
    assert np.array_equal(al.cpu().numpy(), ral) and np.array_equal(nt.cpu().numpy(), rnt)
    assert np.array_equal(tg.cpu().numpy(), ramax)


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3", "bf16_row_pairs"])
@pytest.mark.parametrize("entry", ["packed", "host_lengths"])
def test_bounded_wait_runs_out_and_the_kernel_returns(kv, entry):
    """The tcgen05 kernel's barrier waits are bounded. With a short limit (1e5 cycles, about
    50 us) and the first tile of every CTA's range withheld (sv_inject_wait_timeout), the
    waits for that tile run out: the call returns, the workspace reports SV_ERR_TIMEOUT,
    the kernel ends well before the default limit (about 2 s), and the next calls, on the
    same workspace once its flags are cleared and on a fresh one, match the oracle."""
    import time
    try:
        prev = sv.set_attn_kernel(2)
    except ValueError:
        pytest.skip("tcgen05 kernel not built")
    pairs = kv == "bf16_row_pairs"  # G (1 + D) = 256 rows: the row-pair kernel
    prev_pairs = sv.api.set_row_pairs(1 if pairs else 0)
    try:
        kvd = "bf16" if pairs else kv
        w = synth.Workload("t", B=3, Hq=32 if pairs else 16, Hkv=4, d=128, D=0, T=0, V=8,
                           p=0.5, kv_dtype=kvd, outlier_prob=0.001 if kvd != "bf16" else 0.0)
        x = synth.attn_inputs(w, 23, seq_lens=np.array([900, 5, 300]),
                              draft_len=np.array([7, 0, 3]) + (24 if pairs else 0))
        q, k, v, sc, T, D = dev_attn(x)
        Th = torch.from_numpy(x["seq_lens"].astype(np.int32))
        Dh = torch.from_numpy(x["draft_len"].astype(np.int32))
        md = int(x["draft_len"].max())
        ws = sv.new_workspace(sv.verify_workspace_bytes(sv.api.attn_desc(q, k, 3, md, 900)))
        out = torch.empty_like(q)

        def call(wsp):
            if entry == "packed":
                return sv.spec_verify_attn(q, k, v, T, D, max_draft_len=md, max_seq_len=900,
                                           kv_scale=sc, out=out, workspace=wsp)
            return sv.spec_verify_attn_host_lengths(q, k, v, T, D, Th, Dh, max_draft_len=md,
                                                    max_seq_len=900, kv_scale=sc, out=out,
                                                    workspace=wsp)

        call(ws)  # warm: module load, first launch
        torch.cuda.synchronize()
        assert sv.workspace_status(ws) == 0
        ref = oracle_attn(w, x)
        assert sv.api.inject_wait_timeout(100000) == 0
        t0 = time.perf_counter()
        call(ws)
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
        assert sv.workspace_status(ws, clear=True) == 7   # SV_ERR_TIMEOUT
        assert elapsed < 0.5, elapsed
        assert sv.api.inject_wait_timeout(0) == 0          # the arming was used once
        call(ws)
        torch.cuda.synchronize()
        assert sv.workspace_status(ws) == 0
        assert_close(_bits(out), ref)
        ws2 = sv.new_workspace(sv.verify_workspace_bytes(sv.api.attn_desc(q, k, 3, md, 900)))
        call(ws2)
        torch.cuda.synchronize()
        assert sv.workspace_status(ws2) == 0
        assert_close(_bits(out), ref)
    finally:
        sv.api.inject_wait_timeout(0)
        sv.set_attn_kernel(prev)
        sv.api.set_row_pairs(prev_pairs)
