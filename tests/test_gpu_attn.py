"""GPU parity of spec_verify_attn against the fp64 oracle (max-abs <= 1e-2, normwise
max-rel <= 2e-2): small shapes computed in full (several tiles, ragged tails, edge cases),
the five workloads at full size on sampled (sequence, KV head) units, and device-side
checks."""
import zlib

import numpy as np
import pytest
import torch

import speculative_decoding_verification_gqa_gb300 as sv
from speculative_decoding_verification_gqa_gb300 import synth

from gpu_util import (assert_close, bf16_to_f64, compare, dev_attn, ensure_built, gpu_attn,
                      oracle_attn)

pytestmark = pytest.mark.gpu


def _kernels():
    ensure_built()
    ks = [1]
    prev = sv.api.load_library().sv_set_attn_kernel(2)
    if prev >= 0:
        sv.api.load_library().sv_set_attn_kernel(prev)
        ks.append(2)
    return ks


@pytest.fixture(params=[1, 2], ids=["mma", "tcgen05"])
def kernel(request):
    if request.param not in _kernels():
        pytest.skip("kernel not built")
    prev = sv.set_attn_kernel(request.param)
    yield request.param
    sv.set_attn_kernel(prev)


def _small(B, Hq, Hkv, d, T, D, kv="bf16", seed=0):
    w = synth.Workload("s", B=B, Hq=Hq, Hkv=Hkv, d=d, D=0, T=0, V=8, p=0.5, kv_dtype=kv,
                       outlier_prob=0.001 if kv != "bf16" else 0.0)
    return w, synth.attn_inputs(w, seed, seq_lens=np.array(T), draft_len=np.array(D))


SMALL = {
    "c1": dict(B=1, Hq=4, Hkv=1, d=64, T=(256,), D=(3,)),
    "ragged": dict(B=3, Hq=8, Hkv=2, d=128, T=(1000, 37, 129), D=(5, 0, 15)),
    "decode_D0": dict(B=2, Hq=32, Hkv=8, d=128, T=(300, 777), D=(0, 0)),
    "G1_mha": dict(B=2, Hq=4, Hkv=4, d=128, T=(200, 64), D=(3, 7)),
    "empty_prefix": dict(B=2, Hq=8, Hkv=2, d=64, T=(0, 1), D=(4, 0)),
    "tile_edges": dict(B=4, Hq=8, Hkv=2, d=128, T=(63, 64, 127, 128), D=(0, 1, 0, 1)),
    "rows_136": dict(B=2, Hq=32, Hkv=4, d=128, T=(500, 260), D=(16, 16)),
    "rows_256": dict(B=1, Hq=32, Hkv=4, d=128, T=(400,), D=(31,)),
    "llama3_8b_shape": dict(B=2, Hq=32, Hkv=8, d=128, T=(1500, 333), D=(31, 31)),
    "d64_ragged": dict(B=3, Hq=16, Hkv=2, d=64, T=(513, 5, 2049), D=(8, 2, 1)),
}


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
@pytest.mark.parametrize("name", list(SMALL))
def test_small_shapes_full_oracle(kernel, name, kv):
    w, x = _small(kv=kv, seed=zlib.crc32(name.encode()) % 1000, **SMALL[name])
    got = gpu_attn(x)
    ref = oracle_attn(w, x)
    assert_close(got, ref)


def test_rows_beyond_packed_batch_untouched(kernel):
    w, x = _small(B=2, Hq=8, Hkv=2, d=128, T=(100, 50), D=(3, 2))
    q, k, v, sc, T, D = dev_attn(x)
    rows = q.shape[0]
    qbig = torch.zeros((rows + 5, 8, 128), dtype=torch.bfloat16, device="cuda")
    qbig[:rows] = q
    out = torch.full_like(qbig, 7.0)
    sv.spec_verify_attn(qbig, k, v, T, D, max_draft_len=3, max_seq_len=100, out=out)
    torch.cuda.synchronize()
    assert (out[rows:] == 7.0).all()
    ref = oracle_attn(w, x)
    assert_close(out[:rows].contiguous().view(torch.int16).cpu().numpy().view(np.uint16), ref)


def test_repeatable_and_workspace_reuse(kernel):
    w, x = _small(B=3, Hq=16, Hkv=4, d=128, T=(3000, 10, 900), D=(7, 3, 0))
    q, k, v, sc, T, D = dev_attn(x)
    ws = sv.new_workspace(sv.verify_workspace_bytes(sv.api.attn_desc(q, k, 3, 7, 3000)))
    o1 = sv.spec_verify_attn(q, k, v, T, D, max_draft_len=7, max_seq_len=3000, workspace=ws)
    o2 = sv.spec_verify_attn(q, k, v, T, D, max_draft_len=7, max_seq_len=3000, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)
    assert sv.workspace_status(ws) == 0


def test_device_side_length_check(kernel):
    w, x = _small(B=2, Hq=8, Hkv=2, d=128, T=(100, 50), D=(3, 2))
    q, k, v, sc, T, D = dev_attn(x)
    ws = sv.new_workspace(sv.verify_workspace_bytes(sv.api.attn_desc(q, k, 2, 2, 100)))
    out = torch.full_like(q, 3.0)
    sv.spec_verify_attn(q, k, v, T, D, max_draft_len=2, max_seq_len=100, out=out,
                        workspace=ws)                     # D_0 = 3 > max_draft_len = 2
    assert sv.workspace_status(ws, clear=True) == 8
    assert (out == 3.0).all()
    out2 = sv.spec_verify_attn(q, k, v, T, D, max_draft_len=3, max_seq_len=99, out=out,
                               workspace=ws)              # T_0 = 100 > max_seq_len = 99
    assert sv.workspace_status(ws, clear=True) == 8
    assert (out2 == 3.0).all()
    small_q = q[:5].contiguous()                         # q_rows 5 < sum W = 7
    with pytest.raises(ValueError):
        sv.spec_verify_attn(small_q, k, v, T, D, max_draft_len=3, max_seq_len=100,
                            out=torch.empty_like(q))      # out shape != q shape
    sv.spec_verify_attn(small_q, k, v, T, D, max_draft_len=3, max_seq_len=100, workspace=ws)
    assert sv.workspace_status(ws, clear=True) == 8


# ------------------------------------------------------------------ full-size workloads

_cache = {}


def _full(cfg, D=None):
    key = (cfg, D)
    if key not in _cache:
        _cache.clear()
        w = synth.CONFIGS[cfg]
        if D is None:
            x = synth.attn_inputs(w, 1)
        else:
            T, Dv, _ = synth.lengths(w, 1, D=D)
            x = synth.attn_inputs(w, 1, seq_lens=T, draft_len=Dv)
        _cache[key] = (w, x)
    return _cache[key]


def _sample_units(w, x, n, seed):
    rng = np.random.default_rng(seed)
    B = len(x["seq_lens"])
    picks = {(0, 0), (B - 1, w.Hkv - 1)}
    if w.ragged:  # include the longest and the shortest sequence
        picks.add((int(np.argmax(x["seq_lens"])), 0))
        picks.add((int(np.argmin(x["seq_lens"])), w.Hkv - 1))
    while len(picks) < n:
        picks.add((int(rng.integers(B)), int(rng.integers(w.Hkv))))
    return sorted(picks)


@pytest.mark.parametrize("cfg,D", [("c1", None), ("c2", None), ("c3", None), ("c4", 0),
                                   ("c4", 15), ("c4", 16), ("c4", 31), ("c5", None)])
def test_full_size_sampled_units(kernel, cfg, D):
    w, x = _full(cfg, D)
    got = gpu_attn(x)
    units = None if cfg == "c1" else _sample_units(w, x, 6, seed=7)
    ref = oracle_attn(w, x, units=units)
    ma, mr = assert_close(got, ref)
    # every packed row was written with finite values
    assert np.isfinite(bf16_to_f64(got)).all()
