"""GPU tests of spec_verify_attn_host_lengths: the work plan made on the host from host
copies of the lengths must be the planning kernel's plan, so every output is bit-identical
to spec_verify_attn's (all unit-to-CTA policies, windows, bf16 and FP8), and the oracle
agrees; host-side length errors, the fallback beyond the host plan's capacity, and a
workspace shared with device-planned calls."""
import numpy as np
import pytest
import torch

import speculative_decoding_verification_gqa_gb300 as sv
from speculative_decoding_verification_gqa_gb300 import synth

from gpu_util import assert_close, dev_attn, ensure_built, gpu_attn, oracle_attn

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
    w = synth.Workload("hp", B=B, Hq=Hq, Hkv=Hkv, d=d, D=0, T=0, V=8, p=0.5, kv_dtype=kv,
                       outlier_prob=0.001 if kv != "bf16" else 0.0)
    return w, synth.attn_inputs(w, seed, seq_lens=np.array(T), draft_len=np.array(D))


def gpu_attn_hl(x, *, window=0, workspace=None):
    q, k, v, sc, T, D = dev_attn(x)
    o = sv.spec_verify_attn_host_lengths(
        q, k, v, T, D, torch.from_numpy(x["seq_lens"].astype(np.int32)),
        torch.from_numpy(x["draft_len"].astype(np.int32)),
        max_draft_len=int(x["draft_len"].max()), max_seq_len=int(x["seq_lens"].max()),
        kv_scale=sc, sliding_window=window, workspace=workspace)
    torch.cuda.synchronize()
    return o.view(torch.int16).cpu().numpy().view(np.uint16)


SHAPES = {
    "ragged": dict(B=3, Hq=8, Hkv=2, d=128, T=(1000, 37, 129), D=(5, 0, 15)),
    "rows_256": dict(B=2, Hq=32, Hkv=4, d=128, T=(400, 260), D=(31, 31)),
    "d64": dict(B=3, Hq=16, Hkv=2, d=64, T=(513, 5, 2049), D=(8, 2, 1)),
    "tile_edges": dict(B=4, Hq=8, Hkv=2, d=128, T=(63, 64, 127, 128), D=(0, 1, 0, 1)),
    "c1": dict(B=1, Hq=4, Hkv=1, d=64, T=(256,), D=(3,)),
}


@pytest.mark.parametrize("mode", [-1, 0, 1, 2])
@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
@pytest.mark.parametrize("name", list(SHAPES))
def test_bit_identical_to_the_device_planned_call(kernel, mode, kv, name):
    w, x = _small(kv=kv, seed=5, **SHAPES[name])
    prev = sv.set_unit_ctas(mode)
    try:
        a = gpu_attn(x)
        b = gpu_attn_hl(x)
    finally:
        sv.set_unit_ctas(prev)
    assert np.array_equal(a, b)
    assert_close(b, oracle_attn(w, x))


@pytest.mark.parametrize("W", [1, 100, 4096])
def test_sliding_window(kernel, W):
    w, x = _small(B=3, Hq=8, Hkv=2, d=128, T=(3000, 37, 700), D=(7, 0, 15), seed=6)
    b = gpu_attn_hl(x, window=W)
    assert np.array_equal(b, gpu_attn(x, window=W))
    assert_close(b, oracle_attn(w, x, window=W))


@pytest.mark.parametrize("cfg", ["c2", "c3"])
def test_full_size_workloads(kernel, cfg):
    w = synth.CONFIGS[cfg]
    x = synth.attn_inputs(w, 1)
    b = gpu_attn_hl(x)
    assert np.array_equal(b, gpu_attn(x))
    B = len(x["seq_lens"])
    assert_close(b, oracle_attn(w, x, units=[(0, 0), (B - 1, w.Hkv - 1)]))


def test_beyond_the_host_plan_capacity_plans_on_the_device(kernel):
    """300 sequences (more than a host plan holds): the call plans on the device."""
    rng = np.random.default_rng(8)
    B = 300
    w, x = _small(B=B, Hq=8, Hkv=2, d=128, T=tuple(rng.integers(0, 300, B)),
                  D=tuple(rng.integers(0, 6, B)), seed=8)
    b = gpu_attn_hl(x)
    assert np.array_equal(b, gpu_attn(x))
    assert_close(b, oracle_attn(w, x, units=[(0, 0), (150, 1), (299, 1)]))


def test_lengths_out_of_range_are_reported_on_the_host(kernel):
    w, x = _small(B=2, Hq=8, Hkv=2, d=128, T=(100, 50), D=(3, 2), seed=9)
    q, k, v, sc, T, D = dev_attn(x)
    Th = torch.tensor([100, 50], dtype=torch.int32)
    Dh = torch.tensor([3, 9], dtype=torch.int32)  # beyond max_draft_len
    with pytest.raises(sv.SpecVerifyError) as e:
        sv.spec_verify_attn_host_lengths(q, k, v, T, D, Th, Dh, max_draft_len=3, max_seq_len=100)
    assert e.value.status == 2


def test_workspace_shared_with_device_planned_calls(kernel):
    """Host- and device-planned calls of different shapes alternate on one workspace (the
    combine reads the plan each kind leaves there)."""
    big = dict(B=3, Hq=8, Hkv=2, d=128, T=(5000, 3000, 700), D=(15, 3, 7))
    small = dict(B=2, Hq=8, Hkv=2, d=128, T=(2000, 40), D=(5, 1))
    (w1, x1), (w2, x2) = _small(**big, seed=10), _small(**small, seed=11)
    q, k, *_ = dev_attn(x1)
    desc = sv.api.attn_desc(q, k, 3, 15, 5000)
    ws = sv.new_workspace(sv.verify_workspace_bytes(desc))
    for x in (x1, x2, x1, x2):
        assert np.array_equal(gpu_attn_hl(x, workspace=ws), gpu_attn(x, workspace=ws))
    assert sv.workspace_status(ws) == 0
