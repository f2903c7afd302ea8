"""The verify-attention work plan, computed on the host by the library (sv_plan_preview, the
same plan the planning kernel writes and the host-lengths call passes with its launch),
checked on the CPU against what the plan must be:

* every key a unit's query rows can see lies in the unit's tiles, and no tile lies wholly
  before the first of them or after the last key T_b + D_b (window-causal mask, and the
  sliding window's lower edge: the query at position p sees the W most recent positions,
  "GPU and LLM, chapter 5", "Sliding window");
* every (sequence, KV head, row tile) is one unit, in the documented order;
* the CTA ranges partition the tile line, each within the unit it names, balanced on
  the line with unit starts charged;
* the unit-to-CTA policy: the model's choices on the measured workloads, and forced
  modes.
CPU only: the library loads and plans without a device."""
import itertools

import numpy as np
import pytest

from speculative_decoding_verification_gqa_gb300 import api, build

MT = 128  # query rows per unit


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    return api.load_library()


def _desc(B, Hq, Hkv, d, D, T, fp8=False, W=0, q_rows=None, kv_rows=None):
    return api.AttnDesc(batch=B, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d,
                        max_draft_len=D, max_seq_len=T,
                        q_rows=B * (1 + D) if q_rows is None else q_rows,
                        kv_rows=B * (T + 1 + D) if kv_rows is None else kv_rows,
                        kv_dtype=1 if fp8 else 0, softmax_scale=0.0, sliding_window=W)


def _plan(desc, T, D, sms=152, kernel=2, block_size=0):
    return api.plan_preview(desc, T, D, num_sms=sms, attn_kernel=kernel, block_size=block_size)


def _status(desc, T, D, sms=152, kernel=2, block_size=0, cap=None):
    lib = api.load_library()
    T = np.ascontiguousarray(T, dtype=np.int32)
    D = np.ascontiguousarray(D, dtype=np.int32)
    info = api.PlanInfo()
    if cap is None:
        return lib.sv_plan_preview(desc, block_size, T.ctypes.data, D.ctypes.data, sms, kernel,
                                   info, None, None, None, 0)
    units = np.zeros((max(cap, 1), 4), dtype=np.int32)
    ubeg = np.zeros(cap + 1, dtype=np.int32)
    return lib.sv_plan_preview(desc, block_size, T.ctypes.data, D.ctypes.data, sms, kernel,
                               info, units.ctypes.data, ubeg.ctypes.data, None, cap)


def _visible_keys(T, i, W):
    """Keys the query at position T + i sees: all earlier positions and itself, or the W
    most recent of them."""
    lo = 0 if W == 0 else max(0, T + i - W + 1)
    return lo, T + i


def check_plan(plan, T, D, G, Hkv, W):
    kt = plan["tile_keys"]
    U, TT, C = plan["num_units"], plan["total_tiles"], plan["num_ctas"]
    units, ubeg, cta = plan["units"], plan["unit_begin"], plan["cta_begin"]
    B = len(T)
    nmt = [(G * (1 + int(D[b])) + MT - 1) // MT for b in range(B)]
    # one unit per (b, g, mt), in order
    want = [(b, g, mt) for b in range(B) for g in range(Hkv) for mt in range(nmt[b])]
    if len(set(nmt)) == 1 and nmt[0] > 1:  # row-tile-major
        want = [(b, g, mt) for mt in range(nmt[0]) for b in range(B) for g in range(Hkv)]
    assert U == len(want)
    assert [tuple(u[:3]) for u in units] == want
    # unit tiles: contiguous on the line, covering exactly the keys the rows see
    assert ubeg[0] == 0 and ubeg[U] == TT and np.all(np.diff(ubeg) >= 1)
    for u, (b, g, mt) in enumerate(want):
        Tb, Db = int(T[b]), int(D[b])
        i_first = mt * MT // G
        i_last = min(Db, ((mt + 1) * MT - 1) // G)
        first_key = min(_visible_keys(Tb, i, W)[0] for i in range(i_first, i_last + 1))
        kbase, n = int(units[u][3]), int(ubeg[u + 1] - ubeg[u])
        assert kbase % kt == 0
        assert kbase <= first_key < kbase + kt, (u, kbase, first_key)
        # the last tile holds T_b + D_b (the last key of the sequence's window)
        assert kbase + (n - 1) * kt <= Tb + Db < kbase + n * kt
    # CTA ranges: a partition of the line, each start inside the unit it names
    assert tuple(cta[C]) == (TT, U)
    assert np.all(np.diff(cta[:, 0]) >= 0)
    k = plan["unit_ctas"]
    for c in range(C):
        t, u = int(cta[c, 0]), int(cta[c, 1])
        if k > 0 and c >= U * k:
            assert (t, u) == (TT, U)  # idle CTA
            continue
        assert 0 <= u < U and ubeg[u] <= t < ubeg[u + 1], (c, t, u)
    tiles = np.diff(cta[:, 0])
    if k > 0:
        for u in range(U):  # k equal parts of each unit
            part = tiles[u * k:(u + 1) * k]
            assert part.sum() == ubeg[u + 1] - ubeg[u] and part.max() - part.min() <= 1
            assert np.all(cta[u * k:(u + 1) * k, 1] == u)
    else:
        X = plan["switch_tiles"]
        VT = TT + U * X
        for c in range(C):  # real tiles plus the charge for each unit touched
            t0, t1 = int(cta[c, 0]), int(cta[c + 1, 0])
            touched = len({u for u in range(U) if ubeg[u] < t1 and ubeg[u + 1] > t0})
            assert (t1 - t0) + X * touched <= VT / C + X + 1, (c, t1 - t0, touched)
    return plan


WORKLOADS = {  # name: (B, Hq, Hkv, D, T, fp8)
    "c1": (1, 4, 1, 3, 256, False),
    "c2": (16, 32, 8, 31, 8192, False),
    "c3": (8, 64, 8, 15, 32768, True),
    "c4_d16": (32, 32, 4, 16, 16384, False),
    "c4_d31": (32, 32, 4, 31, 16384, False),
}


@pytest.mark.parametrize("name", sorted(WORKLOADS))
@pytest.mark.parametrize("W", [0, 4096])
def test_uniform_workloads(name, W):
    B, Hq, Hkv, D, T, fp8 = WORKLOADS[name]
    Tv, Dv = [T] * B, [D] * B
    plan = _plan(_desc(B, Hq, Hkv, 128 if name != "c1" else 64, D, T, fp8, W), Tv, Dv)
    check_plan(plan, Tv, Dv, Hq // Hkv, Hkv, W)


def test_policies_chosen_on_the_measured_workloads():
    """The per-tile time model's choices (one CTA per unit on the Llama-3-8B-shaped layer,
    the split line on the 70B-shaped FP8 layer; under a 4096-position window one and two
    CTAs per unit), and the counts of units and tiles."""
    c2 = _plan(_desc(16, 32, 8, 128, 31, 8192), [8192] * 16, [31] * 16)
    assert (c2["num_units"], c2["total_tiles"], c2["unit_ctas"]) == (128, 128 * 65, 1)
    c3 = _plan(_desc(8, 64, 8, 128, 15, 32768, True), [32768] * 8, [15] * 8)
    assert (c3["num_units"], c3["total_tiles"], c3["unit_ctas"]) == (64, 64 * 257, 0)
    w2 = _plan(_desc(16, 32, 8, 128, 31, 8192, W=4096), [8192] * 16, [31] * 16)
    assert w2["unit_ctas"] == 1 and w2["total_tiles"] == 128 * 33
    w3 = _plan(_desc(8, 64, 8, 128, 15, 32768, True, W=4096), [32768] * 8, [15] * 8)
    assert w3["unit_ctas"] == 2 and w3["total_tiles"] == 64 * 33
    # the mma.sync kernel keeps the split line; a paged cache, of small blocks or large,
    # takes the packed layout's choice (the same tile counts)
    assert _plan(_desc(16, 32, 8, 128, 31, 8192), [8192] * 16, [31] * 16,
                 kernel=1)["unit_ctas"] == 0
    for bs in (16, 128):
        assert _plan(_desc(16, 32, 8, 128, 31, 8192), [8192] * 16, [31] * 16,
                     block_size=bs)["unit_ctas"] == 1
        assert _plan(_desc(8, 64, 8, 128, 15, 32768, True), [32768] * 8, [15] * 8,
                     block_size=bs)["unit_ctas"] == 0


@pytest.mark.parametrize("seed", range(12))
def test_ragged_batches(seed):
    """Ragged lengths (the adaptive-draft-length mix: T ~ U[0, 65536], D ~ U{0 .. Dmax}),
    G in {1, 4, 8, 16}, with and without a sliding window, packed or paged, on both
    kernels and on grids smaller than the batch's units."""
    rng = np.random.default_rng(100 + seed)
    G = int(rng.choice([1, 4, 8, 16]))
    Hkv = int(rng.choice([1, 2, 8]))
    Dmax = int(rng.choice([0, 3, 8, 15, 31]))
    nmt_max = (G * (1 + Dmax) + MT - 1) // MT
    B = int(rng.integers(1, min(48, 640 // (Hkv * nmt_max)) + 1))  # the host plan's capacity
    Tv = rng.integers(0, 65537, size=B)
    short = rng.random(B) < 0.2  # some prefixes within the first tiles
    Tv[short] = rng.integers(0, 200, size=int(short.sum()))
    Dv = rng.integers(0, Dmax + 1, size=B)
    W = int(rng.choice([0, 1, 100, 4096, 70000]))
    sms = int(rng.choice([152, 20, 3]))
    kernel = int(rng.choice([1, 2]))
    block_size = int(rng.choice([0, 16, 128, 1024]))  # 0: packed cache
    desc = _desc(B, G * Hkv, Hkv, 128, Dmax, 65536, W=W)
    plan = _plan(desc, Tv, Dv, sms=sms, kernel=kernel, block_size=block_size)
    if block_size and block_size < plan["tile_keys"]:
        assert plan["unit_ctas"] == 0  # small blocks: always the split line
    # a window covering every position of the longest sequence is no window
    W_eff = 0 if W > 65536 + Dmax else W
    check_plan(plan, Tv, Dv, G, Hkv, W_eff)


def test_zero_length_prefixes_and_single_position_windows():
    Tv, Dv = [0, 0, 5, 127, 128, 129], [0, 3, 0, 0, 1, 2]
    for W in (0, 1, 2, 128):
        plan = _plan(_desc(6, 8, 2, 128, 3, 200, W=W), Tv, Dv)
        check_plan(plan, Tv, Dv, 4, 2, W)


@pytest.mark.parametrize("mode", [0, 1, 2, 3, 5])
def test_forced_unit_cta_modes(mode):
    lib = api.load_library()
    prev = lib.sv_set_unit_ctas(mode)
    try:
        for B, sms in ((16, 152), (40, 152), (8, 152)):  # U = 128 (<= C), 320 (> C), 64
            Tv, Dv = [8192] * B, [31] * B
            plan = _plan(_desc(B, 32, 8, 128, 31, 8192), Tv, Dv, sms=sms)
            U, C = plan["num_units"], plan["num_ctas"]
            assert plan["unit_ctas"] == (min(mode, C // U) if U <= C else 0)
            check_plan(plan, Tv, Dv, 4, 8, 0)
    finally:
        lib.sv_set_unit_ctas(prev)


def test_grid_is_capped_by_the_tiles_the_bounds_allow():
    plan = _plan(_desc(1, 4, 1, 64, 3, 256), [256], [3])
    assert plan["num_ctas"] == 3 and plan["num_units"] == 1  # ceil(260 / 128) tiles
    assert plan["num_ctas"] == _plan(_desc(1, 4, 1, 64, 3, 256), [10], [0])["num_ctas"]


def test_rejections():
    d = _desc(4, 32, 8, 128, 7, 1000)
    T, D = [1000] * 4, [7] * 4
    assert _status(d, T, D) == 0
    assert _status(d, [1001, 0, 0, 0], D) == 2          # T_b > max_seq_len
    assert _status(d, T, [8, 0, 0, 0]) == 2             # D_b > max_draft_len
    assert _status(_desc(4, 32, 8, 128, 7, 1000, q_rows=31), T, D) == 2
    assert _status(_desc(4, 32, 8, 128, 7, 1000, kv_rows=4031), T, D) == 2
    # a paged cache: the packed row count does not apply
    assert _status(_desc(4, 32, 8, 128, 7, 1000, kv_rows=0), T, D, block_size=16) == 0
    assert _status(d, T, D, block_size=12) == 2
    assert _status(d, T, D, block_size=4) == 2
    assert _status(d, T, D, sms=0) == 2
    assert _status(d, T, D, kernel=3) == 2
    assert _status(_desc(4, 32, 8, 64, 7, 1000, fp8=True), T, D, kernel=2) == 2
    assert _status(_desc(4, 32, 8, 64, 7, 1000, fp8=True), T, D, kernel=1) == 0
    assert _status(d, T, D, cap=31) == 5                # 32 units
    assert _status(d, T, D, cap=32) == 0
    assert _status(_desc(257, 8, 8, 128, 0, 100), [1] * 257, [0] * 257) == 5
    assert _status(d, T, D, sms=193) == 5
    lib = api.load_library()
    info = api.PlanInfo()
    assert lib.sv_plan_preview(d, 0, None, None, 152, 2, info, None, None, None, 0) == 1
    Tn = np.zeros(4, dtype=np.int32)
    assert lib.sv_plan_preview(d, 0, Tn.ctypes.data, Tn.ctypes.data, 152, 2, None, None, None,
                               None, 0) == 1
    # an empty batch plans nothing
    e = _plan(_desc(0, 32, 8, 128, 7, 1000), [], [])
    assert (e["num_units"], e["total_tiles"]) == (0, 0)


def test_every_small_shape_exhaustively():
    """All batches of up to three sequences with T in a few tile-boundary values and D in
    {0, 1, 31}, for G = 4 and 8, windows 0 and 130."""
    for n in (1, 2, 3):
        for Ts in itertools.product([0, 127, 128, 300], repeat=n):
            for Ds in itertools.product([0, 1, 31], repeat=n):
                for G, W in ((4, 0), (8, 130)):
                    plan = _plan(_desc(n, G * 2, 2, 128, 31, 300, W=W), Ts, Ds, sms=7)
                    check_plan(plan, Ts, Ds, G, 2, W)


def test_row_pair_mode_query(lib):
    """Which calls run the row-pair kernel (sv_row_pair_mode, no device): only when switched
    on, and then when 128 < G (1 + D) <= 256 rows per KV head, bf16, d = 128, packed cache,
    no sliding window, tcgen05, and at most one CTA per (sequence, KV head) per SM."""
    prev = lib.sv_set_row_pairs(0)
    try:
        c4 = lambda D, **kw: _desc(32, 32, 4, 128, D, 16384, **kw)
        assert api.row_pair_mode(c4(31), 152) == 0          # off by default
        assert lib.sv_set_row_pairs(1) == 0
        assert api.row_pair_mode(c4(15), 152) == 0          # 128 rows: one tile
        for D in (16, 23, 31):
            assert api.row_pair_mode(c4(D), 152) == 1       # 136 .. 256 rows
        assert api.row_pair_mode(_desc(32, 64, 4, 128, 31, 16384), 152) == 0  # 512 rows
        assert api.row_pair_mode(c4(16, fp8=True), 152) == 0
        assert api.row_pair_mode(c4(16, W=4096), 152) == 0
        assert api.row_pair_mode(c4(16), 152, block_size=16) == 0
        assert api.row_pair_mode(c4(16), 152, attn_kernel=1) == 0
        assert api.row_pair_mode(_desc(32, 32, 4, 64, 16, 16384), 152) == 0   # d = 64
        assert api.row_pair_mode(c4(16), 127) == 0          # 128 CTAs > 127 SMs
        assert api.row_pair_mode(_desc(4, 32, 4, 128, 31, 1000), 152) == 1   # 16 CTAs
        assert lib.sv_set_row_pairs(0) == 1
        assert api.row_pair_mode(c4(31), 152) == 0
        assert lib.sv_set_row_pairs(2) == -2 and lib.sv_set_row_pairs(-1) == -2
    finally:
        lib.sv_set_row_pairs(prev)


@pytest.mark.parametrize("seed", range(6))
def test_paged_calls_take_the_packed_plan(seed):
    """A paged cache (any block size) gets the packed layout's plan for the same lengths:
    the same units, tile line, unit-to-CTA choice and CTA ranges (the paged and packed
    calls then compute the same tiles, bit for bit)."""
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 40))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.choice([1, 2, 4, 8, 16]))
    Dm = int(rng.integers(0, 32))
    Tm = int(rng.integers(1, 40000))
    Tv = rng.integers(0, Tm + 1, B)
    Dv = rng.integers(0, Dm + 1, B)
    W = int(rng.choice([0, 0, 512, 4096]))
    for fp8 in (False, True):
        desc = _desc(B, Hkv * G, Hkv, 128, Dm, Tm, fp8, W)
        packed = _plan(desc, Tv, Dv)
        for bs in (8, 16, 64, 256):
            paged = _plan(desc, Tv, Dv, block_size=bs)
            for key in ("num_units", "total_tiles", "unit_ctas", "num_ctas"):
                assert paged[key] == packed[key], (bs, key)
            for key in ("units", "unit_begin", "cta_begin"):
                assert np.array_equal(paged[key], packed[key]), (bs, key)
