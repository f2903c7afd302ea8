"""spec_accept_noalloc: the acceptance step for callers that cannot allocate device memory
per call (engines that reserve all device memory at start-up and pass operators only
their inputs and outputs). Its results must equal spec_accept's, bit for bit, on two
calls in a row with different shapes; shapes beyond its fixed scratch are rejected."""
import ctypes

import pytest
import torch

import speculative_decoding_verification_gqa_gb300 as sv
from speculative_decoding_verification_gqa_gb300 import synth

from gpu_util import dev_accept, ensure_built

pytestmark = pytest.mark.gpu

SV_ERR_WORKSPACE = 5


def _noalloc():
    ensure_built()
    f = sv.load_library().spec_accept_noalloc
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    f.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp]
    f.restype = ctypes.c_int
    return f


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def test_noalloc_matches_spec_accept_on_two_calls():
    f = _noalloc()
    stream = torch.cuda.current_stream()
    for cfg, seed in (("c2", 21), ("c5", 22)):
        w = synth.CONFIGS[cfg]
        a = synth.accept_inputs(w, seed)
        lg, dt, dl = dev_accept(a)
        md = int(a["draft_len"].max())
        rows = lg.shape[0]
        ref_tgt = torch.full((rows,), -1, dtype=torch.int32, device="cuda")
        ref_al, ref_nt = sv.spec_accept(lg, dt, dl, max_draft_len=md, target_tokens=ref_tgt)
        B = dl.shape[0]
        al = torch.zeros(B, dtype=torch.int32, device="cuda")
        nt = torch.full((B,), -1, dtype=torch.int32, device="cuda")
        tgt = torch.full((rows,), -1, dtype=torch.int32, device="cuda")
        dtype = 0 if lg.dtype == torch.bfloat16 else 2
        st = f(B, md, w.V, dtype, _p(lg), _p(dt), _p(dl), _p(al), _p(nt), _p(tgt),
               ctypes.c_void_p(stream.cuda_stream))
        assert st == 0
        torch.cuda.synchronize()
        assert torch.equal(al, ref_al) and torch.equal(nt, ref_nt)
        assert torch.equal(tgt, ref_tgt)
        assert (al >= 1).all()


def test_noalloc_rejects_shapes_beyond_its_scratch():
    f = _noalloc()
    t = torch.zeros(4, dtype=torch.int32, device="cuda")
    lg = torch.zeros(4, dtype=torch.float32, device="cuda")
    st = f(70000, 0, 1000, 2, _p(lg), None, _p(t), _p(t), _p(t), None, None)
    assert st == SV_ERR_WORKSPACE


def _check_against_spec_accept(f, a, V):
    lg, dt, dl = dev_accept(a)
    md = int(a["draft_len"].max())
    rows = lg.shape[0]
    ref_tgt = torch.full((rows,), -1, dtype=torch.int32, device="cuda")
    ref_al, ref_nt = sv.spec_accept(lg, dt, dl, max_draft_len=md, target_tokens=ref_tgt)
    B = dl.shape[0]
    al = torch.zeros(B, dtype=torch.int32, device="cuda")
    nt = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    tgt = torch.full((rows,), -1, dtype=torch.int32, device="cuda")
    dtype = 0 if lg.dtype == torch.bfloat16 else 2
    st = f(B, md, V, dtype, _p(lg), _p(dt), _p(dl), _p(al), _p(nt), _p(tgt),
           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    assert torch.equal(al, ref_al) and torch.equal(nt, ref_nt) and torch.equal(tgt, ref_tgt)
    assert (al >= 1).all()


def test_noalloc_rows_beyond_the_finalizing_cta():
    """4,800 window rows (300 sequences of 16): more than the finalizing CTA keeps in shared
    memory, so the target tokens pass through the global part of the fixed scratch, which
    must be left ready for the next call; then a call of the c2 shape."""
    f = _noalloc()
    w = synth.Workload("n", B=300, Hq=1, Hkv=1, d=8, D=15, T=1, V=64, p=0.7)
    _check_against_spec_accept(f, synth.accept_inputs(w, 31), 64)
    w2 = synth.CONFIGS["c2"]
    _check_against_spec_accept(f, synth.accept_inputs(w2, 32), w2.V)


def test_noalloc_largest_accepted_shape_and_the_next():
    """The largest batch of 16-row sequences whose spec_accept workspace fits the fixed
    scratch runs and matches spec_accept twice in a row; one sequence more is rejected with
    SV_ERR_WORKSPACE."""
    f = _noalloc()
    limit = 512 * 1024  # SV_ACCEPT_NOALLOC_MAX_WORKSPACE
    V, D = 48, 15
    lo, hi = 1, 8192
    while lo < hi:  # largest B whose workspace fits
        mid = (lo + hi + 1) // 2
        if sv.accept_workspace_bytes(mid, D, V) <= limit:
            lo = mid
        else:
            hi = mid - 1
    B = lo
    assert sv.accept_workspace_bytes(B + 1, D, V) > limit
    w = synth.Workload("m", B=B, Hq=1, Hkv=1, d=8, D=D, T=1, V=V, p=0.7)
    a = synth.accept_inputs(w, 33)
    assert B * (D + 1) > 30000
    _check_against_spec_accept(f, a, V)
    _check_against_spec_accept(f, synth.accept_inputs(w, 34), V)
    t = torch.zeros(4, dtype=torch.int32, device="cuda")
    lg = torch.zeros(4, dtype=torch.float32, device="cuda")
    st = f(B + 1, D, V, 2, _p(lg), _p(t), _p(t), _p(t), _p(t), None, None)
    assert st == SV_ERR_WORKSPACE
