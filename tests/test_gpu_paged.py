"""GPU parity of spec_verify_attn_paged (verify attention over a block pool found through a
block table): against the paged oracle on small ragged shapes for block sizes below, at
and above the attention tile, with NaN in every unused row and block; bit-identical to the
packed call on the same positions; combined with a sliding window whose reclaimed blocks
have no table entry; device-side checks of the table; the workloads at full size."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_gqa_gb300 as sv
from speculative_decoding_verification_gqa_gb300 import synth

from gpu_util import assert_close, bf16_to_f64, dev_attn, ensure_built, gpu_attn, oracle_attn

pytestmark = pytest.mark.gpu


@pytest.fixture(params=[1, 2], ids=["mma", "tcgen05"])
def kernel(request):
    ensure_built()
    lib = sv.api.load_library()
    prev = lib.sv_set_attn_kernel(request.param)
    if prev < 0:
        pytest.skip("kernel not built")
    yield request.param
    lib.sv_set_attn_kernel(prev)


def _small(B, Hq, Hkv, d, T, D, kv="bf16", seed=0):
    w = synth.Workload("pg", B=B, Hq=Hq, Hkv=Hkv, d=d, D=0, T=0, V=8, p=0.5, kv_dtype=kv,
                       outlier_prob=0.001 if kv != "bf16" else 0.0)
    return w, synth.attn_inputs(w, seed, seq_lens=np.array(T), draft_len=np.array(D))


def _dev_pages(pg, kv_dtype):
    if kv_dtype == "fp8_e4m3":
        k = torch.from_numpy(pg["k_pages"]).cuda()
        v = torch.from_numpy(pg["v_pages"]).cuda()
    else:
        k = torch.from_numpy(pg["k_pages"].view(np.int16)).view(torch.bfloat16).cuda()
        v = torch.from_numpy(pg["v_pages"].view(np.int16)).view(torch.bfloat16).cuda()
    return k, v, torch.from_numpy(pg["block_table"]).cuda()


def gpu_paged(x, pg, *, window=0, workspace=None, table=None):
    q, _, _, sc, T, D = dev_attn(x)
    kp, vp, bt = _dev_pages(pg, "fp8_e4m3" if x["k"].dtype == np.uint8 else "bf16")
    o = sv.spec_verify_attn_paged(q, kp, vp, bt if table is None else table, T, D,
                                  max_draft_len=int(x["draft_len"].max()),
                                  max_seq_len=int(x["seq_lens"].max()), kv_scale=sc,
                                  sliding_window=window, workspace=workspace)
    torch.cuda.synchronize()
    return o.view(torch.int16).cpu().numpy().view(np.uint16)


def same_policy_packed(x, mode=-1):
    """The packed call under the same unit-to-CTA policy as the paged one (by default the
    cost model, which sees the same tile counts): the same tiles, hence the same bits."""
    prev = sv.set_unit_ctas(mode)
    try:
        return gpu_attn(x)
    finally:
        sv.set_unit_ctas(prev)


def paged_oracle(w, x, pg, window=0, units=None):
    return oracle.verify_attn_paged(x["q"], pg["k_pages"], pg["v_pages"], pg["block_table"],
                                    x["seq_lens"], x["draft_len"], Hq=w.Hq, Hkv=w.Hkv, d=w.d,
                                    kv_scale=x["kv_scale"], window=window, units=units)


RAGGED = dict(B=4, Hq=8, Hkv=2, d=128, T=(1000, 37, 300, 2500), D=(5, 0, 15, 9))


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
@pytest.mark.parametrize("bs", [8, 16, 32, 64, 128, 256, 1024])
def test_ragged_batch_against_paged_oracle(kernel, kv, bs):
    w, x = _small(kv=kv, seed=bs, **RAGGED)
    pg = synth.paged_layout(x, bs, seed=bs + 1, spare_blocks=5)
    prev = sv.set_unit_ctas(0)
    try:
        got = gpu_paged(x, pg)
    finally:
        sv.set_unit_ctas(prev)
    assert_close(got, paged_oracle(w, x, pg))
    # the same positions through the packed layout: the same tiles, the same bits
    assert np.array_equal(got, same_policy_packed(x, 0))
    dflt = gpu_paged(x, pg)  # the default policy
    assert_close(dflt, paged_oracle(w, x, pg))
    assert np.array_equal(dflt, same_policy_packed(x))


@pytest.mark.parametrize("d", [64, 128])
def test_head_dim_64_short_and_empty_prefixes(kernel, d):
    w, x = _small(B=3, Hq=16, Hkv=2, d=d, T=(0, 3, 513), D=(4, 2, 1), seed=5)
    pg = synth.paged_layout(x, 16, seed=2, spare_blocks=1)
    assert_close(gpu_paged(x, pg), paged_oracle(w, x, pg))


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
@pytest.mark.parametrize("bs,W", [(16, 40), (16, 300), (64, 129), (256, 100)])
def test_sliding_window_with_reclaimed_blocks(kernel, kv, bs, W):
    """Blocks holding only positions before T - W + 1 are handed back (table entry -1,
    slot NaN): they are never looked up and the result is the windowed one."""
    w, x = _small(B=3, Hq=8, Hkv=2, d=128, T=(700, 260, 90), D=(7, 3, 0), kv=kv, seed=9)
    pg = synth.paged_layout(x, bs, seed=3, spare_blocks=2, reclaim_before_window=W)
    got = gpu_paged(x, pg, window=W)
    assert np.isfinite(bf16_to_f64(got)).all()
    assert_close(got, oracle_attn(w, x, window=W))


def test_table_entry_outside_the_pool_is_reported(kernel):
    """A table entry that must be read but names no block of the pool sets the device-side
    shape flag; the call touches no memory outside the pool."""
    w, x = _small(B=2, Hq=8, Hkv=2, d=128, T=(300, 40), D=(3, 1), seed=4)
    pg = synth.paged_layout(x, 16, seed=4, spare_blocks=0)
    ws = sv.new_workspace(1 << 24)
    for bad in (-1, pg["k_pages"].shape[0], 1 << 30):
        tab = torch.from_numpy(pg["block_table"]).cuda()
        tab[0, 3] = bad
        gpu_paged(x, pg, workspace=ws, table=tab)
        assert sv.workspace_status(ws, clear=True) == 8
    gpu_paged(x, pg, workspace=ws)
    assert sv.workspace_status(ws) == 0


def test_block_table_too_narrow_is_reported(kernel):
    w, x = _small(B=2, Hq=8, Hkv=2, d=128, T=(300, 40), D=(3, 1), seed=6)
    pg = synth.paged_layout(x, 16, seed=5, spare_blocks=0)
    ws = sv.new_workspace(1 << 24)
    narrow = torch.from_numpy(np.ascontiguousarray(pg["block_table"][:, :10])).cuda()
    gpu_paged(x, pg, workspace=ws, table=narrow)  # sequence 0 needs 19 blocks
    assert sv.workspace_status(ws, clear=True) == 8


_cache = {}


def _full(cfg):
    if cfg not in _cache:
        _cache.clear()
        w = synth.CONFIGS[cfg]
        x = synth.attn_inputs(w, 1)
        _cache[cfg] = (w, x, synth.paged_layout(x, 16, seed=11, spare_blocks=64))
    return _cache[cfg]


@pytest.mark.parametrize("cfg", ["c2", "c3"])
def test_full_size_16_position_blocks(kernel, cfg):
    """The workloads with 16-position blocks scattered over the pool: bit-identical to the
    packed call under the same policy (c2: one CTA per unit, c3: the split tile line), and
    the oracle on sampled units."""
    w, x, pg = _full(cfg)
    got = gpu_paged(x, pg)
    assert np.array_equal(got, same_policy_packed(x))
    B = len(x["seq_lens"])
    units = [(0, 0), (B - 1, w.Hkv - 1), (B // 2, 1)]
    assert_close(got, oracle_attn(w, x, units=units))


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_paged_under_every_unit_cta_policy(kernel, mode):
    """Forced unit-to-CTA policies apply to paged calls too, and give the packed call's
    bits under the same policy."""
    w, x = _small(kv="bf16", seed=19, **RAGGED)
    pg = synth.paged_layout(x, 16, seed=20, spare_blocks=2)
    prev = sv.set_unit_ctas(mode)
    try:
        got = gpu_paged(x, pg)
    finally:
        sv.set_unit_ctas(prev)
    assert_close(got, paged_oracle(w, x, pg))
    assert np.array_equal(got, same_policy_packed(x, mode))
