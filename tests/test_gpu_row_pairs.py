"""GPU parity of the row-pair kernel (one CTA per (sequence, KV head) holding both 128-row
tiles of its G (1 + D) query rows when 128 < G (1 + D) <= 256, each K/V tile read once for
both) against the fp64 oracle: shapes with two row tiles, with one and two in the same
batch, G = 8 and 16, tile edges, NaN rows past the cache, device-side length checks, and
agreement with the unit plan and with the host-lengths call."""
import numpy as np
import pytest
import torch

import speculative_decoding_verification_gqa_gb300 as sv
from speculative_decoding_verification_gqa_gb300 import synth

from gpu_util import assert_close, bf16_to_f64, dev_attn, ensure_built, gpu_attn, oracle_attn

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def tcgen05():
    ensure_built()
    try:
        prev = sv.set_attn_kernel(2)
    except ValueError:
        pytest.skip("tcgen05 kernel not built")
    yield
    sv.set_attn_kernel(prev)
    sv.api.set_row_pairs(0)


def _small(B, Hq, Hkv, T, D, d=128, seed=0):
    w = synth.Workload("p", B=B, Hq=Hq, Hkv=Hkv, d=d, D=0, T=0, V=8, p=0.5)
    return w, synth.attn_inputs(w, seed, seq_lens=np.array(T), draft_len=np.array(D))


CASES = {
    "rows_136": dict(B=2, Hq=32, Hkv=4, T=(500, 260), D=(16, 16)),
    "rows_192": dict(B=2, Hq=32, Hkv=4, T=(700, 129), D=(23, 23)),
    "rows_256": dict(B=1, Hq=32, Hkv=4, T=(400,), D=(31,)),
    # row tiles per sequence: 2, 1, 2, 1 (the second row tile of 128-row sequences is idle)
    "one_and_two_tiles": dict(B=4, Hq=32, Hkv=4, T=(1000, 37, 129, 0), D=(31, 15, 16, 0)),
    "G16": dict(B=3, Hq=64, Hkv=4, T=(300, 2, 1025), D=(8, 15, 0)),
    "tile_edges": dict(B=4, Hq=16, Hkv=2, T=(127, 128, 255, 0), D=(16, 17, 31, 20)),
    "long": dict(B=2, Hq=32, Hkv=4, T=(9000, 4000), D=(31, 20)),
}


def _applies(x, Hq, Hkv):
    q = torch.empty((1, Hq, 128), dtype=torch.bfloat16)
    k = torch.empty((1, Hkv, 128), dtype=torch.bfloat16)
    desc = sv.api.attn_desc(q, k, len(x["seq_lens"]), int(x["draft_len"].max()),
                            int(x["seq_lens"].max()))
    return sv.api.row_pair_mode(desc, torch.cuda.get_device_properties(0).multi_processor_count)


@pytest.mark.parametrize("name", list(CASES))
def test_row_pairs_match_the_oracle(name):
    c = CASES[name]
    w, x = _small(seed=len(name), **c)
    ref = oracle_attn(w, x)
    sv.api.set_row_pairs(1)
    assert _applies(x, c["Hq"], c["Hkv"]) == 1
    got = gpu_attn(x)
    assert np.isfinite(bf16_to_f64(got)).all()
    assert_close(got, ref)
    sv.api.set_row_pairs(0)
    assert _applies(x, c["Hq"], c["Hkv"]) == 0
    assert_close(gpu_attn(x), ref)  # the unit plan on the same inputs


def test_row_pairs_nan_rows_after_the_last_sequence():
    """The last tile of the last sequence overlaps NaN rows past the packed cache; the V rows
    past the sequence's end are cleared before both row tiles' P V read them."""
    w, x = _small(B=2, Hq=32, Hkv=4, T=(300, 190), D=(20, 31), seed=4)
    pad = 200
    for n in ("k", "v"):
        a = x[n]
        x[n] = np.concatenate([a, np.full((pad,) + a.shape[1:], 0x7FC0, dtype=a.dtype)])
    sv.api.set_row_pairs(1)
    got = gpu_attn(x)
    assert np.isfinite(bf16_to_f64(got)).all()
    assert_close(got, oracle_attn(w, x))


def test_row_pairs_host_lengths_call_is_the_same_kernel():
    w, x = _small(B=3, Hq=32, Hkv=4, T=(2000, 5, 700), D=(31, 17, 24), seed=9)
    q, k, v, sc, T, D = dev_attn(x)
    Th = torch.from_numpy(x["seq_lens"].astype(np.int32))
    Dh = torch.from_numpy(x["draft_len"].astype(np.int32))
    sv.api.set_row_pairs(1)
    a = sv.spec_verify_attn(q, k, v, T, D, max_draft_len=31, max_seq_len=2000)
    b = sv.spec_verify_attn_host_lengths(q, k, v, T, D, Th, Dh, max_draft_len=31,
                                         max_seq_len=2000)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert_close(b.view(torch.int16).cpu().numpy().view(np.uint16), oracle_attn(w, x))


def test_row_pairs_repeatable_and_device_side_checks():
    w, x = _small(B=2, Hq=32, Hkv=4, T=(100, 50), D=(20, 17), seed=11)
    q, k, v, sc, T, D = dev_attn(x)
    sv.api.set_row_pairs(1)
    ws = sv.new_workspace(sv.verify_workspace_bytes(sv.api.attn_desc(q, k, 2, 20, 100)))
    o1 = sv.spec_verify_attn(q, k, v, T, D, max_draft_len=20, max_seq_len=100, workspace=ws)
    o2 = sv.spec_verify_attn(q, k, v, T, D, max_draft_len=20, max_seq_len=100, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and sv.workspace_status(ws) == 0
    out = torch.full_like(q, 3.0)
    sv.spec_verify_attn(q, k, v, T, D, max_draft_len=20, max_seq_len=99, out=out,
                        workspace=ws)                      # T_0 = 100 > max_seq_len = 99
    assert sv.workspace_status(ws, clear=True) == 8
    assert (out == 3.0).all()
    small_k = k[:100].contiguous()                          # kv_rows 100 < sum (T + W)
    sv.spec_verify_attn(q, small_k, small_k, T, D, max_draft_len=20, max_seq_len=100,
                        out=out, workspace=ws)
    assert sv.workspace_status(ws, clear=True) == 8
    assert (out == 3.0).all()


@pytest.mark.parametrize("D", [16, 23, 31])
def test_full_size_tile_sweep_row_pairs_and_unit_plan(D):
    """The tile sweep's workload (B = 32, Hkv = 4, G = 8, T = 16384) with two row tiles:
    sampled units of the row-pair kernel and of the unit plan against the oracle."""
    w = synth.CONFIGS["c4"]
    T, Dv, _ = synth.lengths(w, 1, D=D)
    x = synth.attn_inputs(w, 1, seq_lens=T, draft_len=Dv)
    sv.api.set_row_pairs(1)
    assert _applies(x, w.Hq, w.Hkv) == 1
    units = [(0, 0), (31, 3), (7, 1), (19, 2), (25, 0)]
    ref = oracle_attn(w, x, units=units)
    assert_close(gpu_attn(x), ref)
    sv.api.set_row_pairs(0)
    assert_close(gpu_attn(x), ref)
