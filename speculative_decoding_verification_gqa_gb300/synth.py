"""Seeded synthetic inputs for the verification step (host, numpy).

This module only draws and encodes inputs; it holds none of the attention or
acceptance arithmetic. Both the CUDA path and the fp64 oracle consume what it returns.

Recipes (one per workload; see ``CONFIGS``):

* Q, K, V: N(0, 1) float32 samples rounded to bfloat16 (round-to-nearest-even).
* FP8 K/V: N(0, 1) samples, each element multiplied by 20 with probability 0.001
  (outliers), then quantised to OCP E4M3 codes with a per-KV-head fp32 scale
  absmax / 448 (absmax over every batch row and position of that head), rounding to
  nearest even. The scales are returned as ``kv_scale [2, Hkv]`` (K first, then V).
* Logits: N(0, 1) samples, stored as fp32 or rounded to bf16.
* Draft tokens: at each of the D_b positions, independently, with probability p the
  draft equals the target's greedy token for that row (numpy's first-occurrence argmax,
  so ties go to the lowest index), otherwise a token drawn uniformly from the V - 1 other
  ids. An id that merely ties the maximum therefore counts as a mismatch.
* Ragged batches: T_b uniform on [1024, 65536], D_b uniform on {1, 2, 4, 8} and a match
  probability p_b uniform on (0.4, 0.9) per sequence; sequences are packed back to back.
* Paged caches (``paged_layout``): the packed K/V rows of each sequence cut into blocks of
  ``block_size`` positions, the blocks placed at seeded random physical slots of a pool
  that also holds spare blocks; unused rows (the tail of each sequence's last block, spare
  blocks) hold a fill pattern (NaN by default) and unused block-table entries are -1.

Streams: every array is drawn from its own ``SeedSequence(seed, spawn_key=(tag, chunk))``
so that results do not depend on the number of threads used to draw them.
"""
from __future__ import annotations

import concurrent.futures as cf
import dataclasses
import os
from typing import Optional, Sequence

import numpy as np

# stream tags
_TAG_Q, _TAG_K, _TAG_V, _TAG_LOGITS, _TAG_DRAFT, _TAG_LENS, _TAG_OUTLIER = range(1, 8)
_CHUNK = 1 << 22  # samples per independently seeded chunk


@dataclasses.dataclass(frozen=True)
class Workload:
    """One verification workload. ``T`` / ``D`` are per-sequence constants unless
    ``ragged`` is set, in which case they are drawn per sequence."""
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    D: int
    T: int
    V: int
    p: float
    kv_dtype: str = "bf16"          # "bf16" or "fp8_e4m3"
    logits_dtype: str = "bf16"      # "bf16" or "fp32"
    ragged: bool = False
    T_range: tuple = (1024, 65536)
    D_choices: tuple = (1, 2, 4, 8)
    p_range: tuple = (0.4, 0.9)
    outlier_prob: float = 0.0
    outlier_mult: float = 20.0

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


CONFIGS = {
    # tiny verify step
    "c1": Workload("c1-tiny", B=1, Hq=4, Hkv=1, d=64, D=3, T=256, V=1000, p=0.7,
                   logits_dtype="fp32"),
    # Llama-3-8B-shaped layer: G*(1+D) = 128
    "c2": Workload("c2-llama3-8b", B=16, Hq=32, Hkv=8, d=128, D=31, T=8192, V=128256,
                   p=0.8),
    # Llama-3.1-70B-shaped layer, FP8 E4M3 KV with per-head scales
    "c3": Workload("c3-llama31-70b-fp8kv", B=8, Hq=64, Hkv=8, d=128, D=15, T=32768,
                   V=128256, p=0.75, kv_dtype="fp8_e4m3", outlier_prob=0.001),
    # tile-boundary sweep, D in {0,1,3,7,15,16,23,31}
    "c4": Workload("c4-tile-sweep", B=32, Hq=32, Hkv=4, d=128, D=15, T=16384, V=32000,
                   p=0.7),
    # ragged adaptive-gamma batch
    "c5": Workload("c5-ragged", B=64, Hq=32, Hkv=8, d=128, D=8, T=65536, V=128256,
                   p=0.65, ragged=True),
}
C4_SWEEP_D = (0, 1, 3, 7, 15, 16, 23, 31)


def _ss(seed: int, tag: int, chunk: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(
        np.random.SeedSequence(int(seed), spawn_key=(int(tag), int(chunk)))))


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + rounding) >> np.uint32(16)).astype(np.uint16)


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def _normal_bf16(n: int, seed: int, tag: int) -> np.ndarray:
    """n N(0,1) samples as bf16 bits, drawn in independently seeded chunks in parallel."""
    out = np.empty(n, dtype=np.uint16)
    chunks = [(c, c * _CHUNK, min(n, (c + 1) * _CHUNK)) for c in range((n + _CHUNK - 1) // _CHUNK)]

    def work(arg):
        c, lo, hi = arg
        out[lo:hi] = bf16_bits(_ss(seed, tag, c).standard_normal(hi - lo, dtype=np.float32))

    if len(chunks) <= 1:
        for ch in chunks:
            work(ch)
    else:
        with cf.ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(work, chunks))
    return out


def _normal_f32(n: int, seed: int, tag: int) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    chunks = [(c, c * _CHUNK, min(n, (c + 1) * _CHUNK)) for c in range((n + _CHUNK - 1) // _CHUNK)]

    def work(arg):
        c, lo, hi = arg
        out[lo:hi] = _ss(seed, tag, c).standard_normal(hi - lo, dtype=np.float32)

    with cf.ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(work, chunks))
    return out


def e4m3_codes(x: np.ndarray) -> np.ndarray:
    """float32 -> OCP E4M3 codes (uint8), round to nearest even, via torch's
    float8_e4m3fn cast. Inputs must already lie within [-448, 448]."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def lengths(w: Workload, seed: int, D: Optional[int] = None):
    """Per-sequence (seq_lens T_b, draft_len D_b, match probability p_b)."""
    if w.ragged:
        g = _ss(seed, _TAG_LENS)
        T = g.integers(w.T_range[0], w.T_range[1] + 1, size=w.B).astype(np.int32)
        Dv = np.asarray(w.D_choices, dtype=np.int32)[g.integers(0, len(w.D_choices), size=w.B)]
        p = g.uniform(w.p_range[0], w.p_range[1], size=w.B)
        return T, Dv.astype(np.int32), p
    Dc = w.D if D is None else D
    return (np.full(w.B, w.T, dtype=np.int32), np.full(w.B, Dc, dtype=np.int32),
            np.full(w.B, w.p, dtype=np.float64))


def attn_inputs(w: Workload, seed: int, seq_lens=None, draft_len=None):
    """Returns dict(q, k, v, kv_scale, seq_lens, draft_len).

    q: uint16 bf16 bits [sum W, Hq, d]; k, v: uint16 bf16 bits or uint8 E4M3 codes
    [sum (T + W), Hkv, d]; kv_scale: float32 [2, Hkv] (None for bf16)."""
    if seq_lens is None or draft_len is None:
        T, Dv, _ = lengths(w, seed)
        seq_lens = T if seq_lens is None else seq_lens
        draft_len = Dv if draft_len is None else draft_len
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    draft_len = np.asarray(draft_len, dtype=np.int32)
    rows = int(np.sum(draft_len.astype(np.int64) + 1))
    kv_rows = int(np.sum(seq_lens.astype(np.int64) + draft_len + 1))
    q = _normal_bf16(rows * w.Hq * w.d, seed, _TAG_Q).reshape(rows, w.Hq, w.d)
    n_kv = kv_rows * w.Hkv * w.d
    if w.kv_dtype == "bf16":
        k = _normal_bf16(n_kv, seed, _TAG_K).reshape(kv_rows, w.Hkv, w.d)
        v = _normal_bf16(n_kv, seed, _TAG_V).reshape(kv_rows, w.Hkv, w.d)
        scale = None
    elif w.kv_dtype == "fp8_e4m3":
        arrs, scales = [], []
        for tag, otag in ((_TAG_K, _TAG_OUTLIER), (_TAG_V, _TAG_OUTLIER + 16)):
            x = _normal_f32(n_kv, seed, tag)
            if w.outlier_prob > 0:
                hit = _ss(seed, otag).random(n_kv, dtype=np.float32) < np.float32(w.outlier_prob)
                x[hit] *= np.float32(w.outlier_mult)
            x = x.reshape(kv_rows, w.Hkv, w.d)
            absmax = np.abs(x).max(axis=(0, 2)).astype(np.float32)
            s = (absmax / np.float32(448.0)).astype(np.float32)
            s[s == 0] = np.float32(1.0)
            arrs.append(e4m3_codes(x / s[None, :, None]))
            scales.append(s)
            del x
        k, v = arrs
        scale = np.stack(scales).astype(np.float32)
    else:
        raise ValueError(w.kv_dtype)
    return dict(q=q, k=k, v=v, kv_scale=scale, seq_lens=seq_lens, draft_len=draft_len)


def accept_inputs(w: Workload, seed: int, draft_len=None, p=None):
    """Returns dict(logits, draft_tokens, draft_len, p).

    logits: float32 [sum W, V] or uint16 bf16 bits; draft_tokens int32 [sum D]."""
    if draft_len is None or p is None:
        _, Dv, pv = lengths(w, seed)
        draft_len = Dv if draft_len is None else draft_len
        p = pv if p is None else p
    draft_len = np.asarray(draft_len, dtype=np.int32)
    p = np.broadcast_to(np.asarray(p, dtype=np.float64), draft_len.shape)
    rows = int(np.sum(draft_len.astype(np.int64) + 1))
    x = _normal_f32(rows * w.V, seed, _TAG_LOGITS).reshape(rows, w.V)
    if w.logits_dtype == "bf16":
        logits = bf16_bits(x)
        ref = logits.astype(np.uint32) << np.uint32(16)
        greedy = np.argmax(ref.view(np.float32), axis=1)
    elif w.logits_dtype == "fp32":
        logits = x
        greedy = np.argmax(x, axis=1)
    else:
        raise ValueError(w.logits_dtype)
    del x
    g = _ss(seed, _TAG_DRAFT)
    drafts = []
    q_off = 0
    for b, D in enumerate(draft_len.tolist()):
        for j in range(D):
            tgt = int(greedy[q_off + j])
            if g.random() < p[b] or w.V == 1:
                drafts.append(tgt)
            else:
                o = int(g.integers(0, w.V - 1))
                drafts.append(o if o < tgt else o + 1)
        q_off += D + 1
    return dict(logits=logits, draft_tokens=np.asarray(drafts, dtype=np.int32),
                draft_len=draft_len, p=np.asarray(p))


_TAG_DRAFT_LOGITS, _TAG_UNIFORM = 51, 52


def stochastic_inputs(w: Workload, seed: int, draft_len=None, noise: float = 0.7):
    """Inputs of sampled-decoding acceptance: the target's logits of every window row (those
    of accept_inputs), the drafter's logits at every draft position (the target's row of
    that position plus N(0, noise^2) per entry, in the logits' dtype: a drafter that mostly
    agrees), the drafted tokens (the drafter row's argmax with the sequence's match
    probability p, else a uniform token), and uniform draws u_accept [sum D] and u_sample
    [B] in [0, 1). Returns dict(target_logits, draft_logits, draft_tokens, draft_len,
    u_accept, u_sample)."""
    a = accept_inputs(w, seed, draft_len=draft_len)
    Dv = a["draft_len"]
    tgt = a["logits"]
    rows = [int(o) + j for o, D in zip(np.concatenate([[0], np.cumsum(Dv + 1)[:-1]]), Dv)
            for j in range(int(D))]
    nd = len(rows)
    t32 = (tgt[rows].astype(np.uint32) << np.uint32(16)).view(np.float32) \
        if tgt.dtype == np.uint16 else tgt[rows]
    drf = t32 + noise * _normal_f32(nd * w.V, seed, _TAG_DRAFT_LOGITS).reshape(nd, w.V)
    if tgt.dtype == np.uint16:
        drf = bf16_bits(drf)
        greedy = np.argmax((drf.astype(np.uint32) << np.uint32(16)).view(np.float32), axis=1) \
            if nd else np.zeros(0, np.int64)
    else:
        drf = drf.astype(np.float32)
        greedy = np.argmax(drf, axis=1) if nd else np.zeros(0, np.int64)
    g = _ss(seed, _TAG_UNIFORM)
    p = np.repeat(np.asarray(a["p"], dtype=np.float64), Dv)
    other = g.integers(0, w.V, size=nd)
    toks = np.where(g.random(nd) < p, greedy, other).astype(np.int32)
    return dict(target_logits=tgt, draft_logits=drf.reshape(nd, w.V), draft_tokens=toks,
                draft_len=Dv, u_accept=g.random(nd, dtype=np.float32),
                u_sample=g.random(len(Dv), dtype=np.float32))


def packed_offsets(seq_lens: Sequence[int], draft_len: Sequence[int]):
    """Start rows of each sequence in the packed q/out and k/v arrays (host-side
    bookkeeping for callers that build packed batches)."""
    W = np.asarray(draft_len, dtype=np.int64) + 1
    KV = np.asarray(seq_lens, dtype=np.int64) + W
    return (np.concatenate([[0], np.cumsum(W)]), np.concatenate([[0], np.cumsum(KV)]))


_TAG_PAGES = 41


def paged_layout(x, block_size: int, seed: int, spare_blocks: int = 3, fill: str = "nan",
                 reclaim_before_window: int = 0):
    """Moves the packed K/V of ``attn_inputs`` into a paged pool.

    Returns dict(k_pages, v_pages, block_table, block_size): k_pages, v_pages
    [num_blocks, block_size, Hkv, d] (the packed arrays' dtype); block_table int32
    [B, max_blocks] where logical block n of sequence b (positions n*block_size ..) lives
    in physical block block_table[b, n]; entries past a sequence's last block are -1.
    With reclaim_before_window = W > 0, blocks holding only positions before T_b - W + 1
    (outside every window row's sliding window) are given back to the pool: their entries
    are -1 and their slots hold the fill pattern."""
    if block_size < 1:
        raise ValueError("block_size must be >= 1")
    k, v = x["k"], x["v"]
    T = np.asarray(x["seq_lens"], dtype=np.int64)
    R = T + np.asarray(x["draft_len"], dtype=np.int64) + 1  # cache rows per sequence
    nblk = (R + block_size - 1) // block_size
    used = int(nblk.sum())
    num_blocks = used + int(spare_blocks)
    perm = _ss(seed, _TAG_PAGES).permutation(num_blocks)
    Hkv, d = k.shape[1], k.shape[2]
    if k.dtype == np.uint8:
        pat = {"nan": 0x7F, "zero": 0}[fill]
    else:
        pat = {"nan": 0x7FC0, "zero": 0}[fill]
    kp = np.full((num_blocks, block_size, Hkv, d), pat, dtype=k.dtype)
    vp = np.full((num_blocks, block_size, Hkv, d), pat, dtype=v.dtype)
    table = np.full((len(T), max(int(nblk.max()) if len(T) else 1, 1)), -1, dtype=np.int32)
    row0 = 0
    nxt = 0
    for b in range(len(T)):
        first_kept = 0
        if reclaim_before_window > 0:
            first_kept = max(int(T[b]) - reclaim_before_window + 1, 0) // block_size
        for n in range(int(nblk[b])):
            phys = int(perm[nxt])
            nxt += 1
            if n < first_kept:
                continue  # reclaimed: the slot keeps the fill pattern
            lo = n * block_size
            hi = min(lo + block_size, int(R[b]))
            kp[phys, :hi - lo] = k[row0 + lo:row0 + hi]
            vp[phys, :hi - lo] = v[row0 + lo:row0 + hi]
            table[b, n] = phys
        row0 += int(R[b])
    return dict(k_pages=kp, v_pages=vp, block_table=table, block_size=block_size)
