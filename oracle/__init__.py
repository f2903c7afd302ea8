"""fp64 CPU oracle for the speculative-decoding verification step.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this package. The CUDA library never imports, links or
calls it, and it shares no code with the CUDA library.

The arithmetic lives in ``oracle.c`` (plain C, fp64, OpenMP over independent output
rows); this module compiles it with gcc on first use and marshals numpy arrays.

Functions and the passages they follow (page title, then section):

* ``verify_attn`` -- GQA verify attention with a window-causal mask and a materialised
  softmax. "GPU and LLM, chapter 5": "GQA", "FlashAttention" (attention =
  softmax(Q K^T) V) and "Speculative decoding (2)" (one forward over the 1+D positions).
* ``verify_attn_online`` -- the same result through the online-softmax update of
  "GPU and LLM, chapter 5", "Online softmax: carry the max and the sum".
* ``verify_attn(window=W)`` -- sliding-window verify attention: "GPU and LLM, chapter 5",
  "Sliding window: do not keep the distant past" (each position sees the W most recent
  positions, itself included).
* ``verify_attn_paged`` -- the same attention over a paged cache: "GPU and LLM, chapter
  5", "PagedAttention (2): manage with fixed-size pages" (fixed-size blocks of positions
  anywhere in memory, found through a per-sequence block table). The rows are gathered
  back into the packed layout, then ``verify_attn`` runs on them.
* ``argmax_rows`` -- naive first-index argmax (target's greedy choice per window row).
* ``accept`` -- first-mismatch acceptance: "Co-Designing AI Models Using Speculative
  Decoding" summary, "basic structure" (AL in [1, 1+D]); "GPU and LLM, chapter 5",
  "Speculative decoding (2)" (the target's own token replaces the first rejected draft).
* ``draft_signals`` -- per row, the confidence (largest softmax probability) and the
  entropy (nats) of the softmax: "SpecKV" summary, "technical core", item 1.
* ``accept_stochastic`` -- distribution-preserving acceptance: "GPU and LLM, chapter 5",
  "Speculative decoding (2)" (the acceptance rule leaves the output distribution that of
  the large model alone); the rule of the paper that page cites (Leviathan et al., 2023):
  keep draft x with probability min(1, p(x)/q(x)), at the first rejection draw from the
  normalised max(0, p - q), with every draft kept draw from the target's last row.
* ``stochastic_decisions`` -- every keep / reject decision of that rule as a signed
  relative margin (positive: kept), also at positions after the first rejection, so a
  test can check another implementation's path decision by decision.
* ``bf16_to_f64`` / ``e4m3_to_f64`` -- decoders written from the binary32 and OCP E4M3
  format definitions.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` next to it (gcc, OpenMP, no FMA
    contraction so results do not depend on the host's vector unit)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            p = ctypes.c_void_p
            i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.orc_bf16_to_f64.restype = dbl
            lib.orc_e4m3_to_f64.argtypes = [ctypes.c_uint8]
            lib.orc_e4m3_to_f64.restype = dbl
            lib.orc_num_threads.restype = i32
            attn = [i32, i32, i32, i32, p, p, i32, p, p, p, p, dbl, p, p, p, i32]
            lib.orc_verify_attn.argtypes = attn + [i32]
            lib.orc_verify_attn.restype = i32
            lib.orc_verify_attn_online.argtypes = attn + [i32, i32]
            lib.orc_verify_attn_online.restype = i32
            lib.orc_argmax_rows.argtypes = [i64, i64, i32, p, p, i32]
            lib.orc_argmax_rows.restype = i32
            lib.orc_accept.argtypes = [i32, p, p, p, p, p]
            lib.orc_accept.restype = i32
            lib.orc_draft_signals.argtypes = [i64, i64, i32, p, p, p, i32]
            lib.orc_draft_signals.restype = i32
            lib.orc_accept_stochastic.argtypes = [i32, i64, i32, p, p, p, p, p, p, dbl, p, p, p,
                                                  p]
            lib.orc_accept_stochastic.restype = i32
            lib.orc_stochastic_decisions.argtypes = [i32, i64, i32, p, p, p, p, p, dbl, p]
            lib.orc_stochastic_decisions.restype = i32
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return _load().orc_num_threads()


def bf16_to_f64(bits: int) -> float:
    return _load().orc_bf16_to_f64(int(bits))


def e4m3_to_f64(bits: int) -> float:
    return _load().orc_e4m3_to_f64(int(bits))


def _attn_args(q, k, v, seq_lens, draft_len, kv_scale, Hq, Hkv, d, scale, units, rows_sel):
    q = np.ascontiguousarray(q, dtype=np.uint16)
    fp8 = k.dtype == np.uint8
    k = np.ascontiguousarray(k)
    v = np.ascontiguousarray(v)
    if k.dtype != v.dtype or k.dtype not in (np.uint8, np.uint16):
        raise TypeError("k and v must both be uint16 (bf16 bits) or uint8 (e4m3 codes)")
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    draft_len = np.ascontiguousarray(draft_len, dtype=np.int32)
    B = seq_lens.shape[0]
    if kv_scale is not None:
        kv_scale = np.ascontiguousarray(kv_scale, dtype=np.float32).reshape(2, Hkv)
    elif fp8:
        raise ValueError("fp8 k/v need kv_scale")
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    mask = None
    if units is not None:
        mask = np.zeros(B * Hkv, dtype=np.uint8)
        for (b, g) in units:
            mask[b * Hkv + g] = 1
    rows = int(np.sum(draft_len.astype(np.int64) + 1))
    rmask = None
    if rows_sel is not None:
        rmask = np.ascontiguousarray(rows_sel, dtype=np.uint8).reshape(-1)
        if rmask.size != rows * Hq:
            raise ValueError("row selection must have sum(1 + D_b) * Hq entries")
    kv_rows = int(np.sum(seq_lens.astype(np.int64) + draft_len + 1))
    if q.size != rows * Hq * d or k.size < kv_rows * Hkv * d or v.size < kv_rows * Hkv * d:
        raise ValueError("array sizes do not match seq_lens / draft_len")
    return q, k, v, seq_lens, draft_len, kv_scale, float(scale), mask, rmask, fp8, B, rows


def verify_attn(q, k, v, seq_lens, draft_len, *, Hq, Hkv, d, kv_scale=None, scale=None,
                units=None, rows=None, nthreads=0, online_tile=0, out=None, window=0):
    """fp64 verify attention. q: bf16 bits [sum W, Hq, d]; k, v: bf16 bits or e4m3 codes
    [sum (T+W), Hkv, d]. Returns fp64 [sum W, Hq, d]. ``units`` (an iterable of
    (b, kv_head)) and ``rows`` (a bool array [sum W, Hq]) restrict the outputs computed;
    the others are NaN. ``window`` = 0 lets window row i see keys 0 .. T+i; a sliding
    window of W >= 1 positions keeps only keys max(0, T+i-W+1) .. T+i."""
    (q, k, v, seq_lens, draft_len, kv_scale, scale, mask, rmask, fp8, B,
     rows) = _attn_args(q, k, v, seq_lens, draft_len, kv_scale, Hq, Hkv, d, scale, units,
                        rows)
    if out is None:
        out = np.full((rows, Hq, d), np.nan, dtype=np.float64)
    lib = _load()
    args = [B, Hq, Hkv, d, _ptr(seq_lens), _ptr(draft_len), int(fp8), _ptr(q), _ptr(k),
            _ptr(v), _ptr(kv_scale), scale, _ptr(mask), _ptr(rmask), _ptr(out), int(nthreads)]
    if window < 0:
        raise ValueError("window must be >= 0")
    if online_tile:
        rc = lib.orc_verify_attn_online(*args, int(online_tile), int(window))
    else:
        rc = lib.orc_verify_attn(*args, int(window))
    if rc:
        raise ValueError("oracle rejected the arguments")
    return out


def verify_attn_paged(q, k_pages, v_pages, block_table, seq_lens, draft_len, *, Hq, Hkv, d,
                      kv_scale=None, window=0, **kw):
    """fp64 verify attention over a paged cache. k_pages, v_pages: [num_blocks, block_size,
    Hkv, d] (bf16 bits or e4m3 codes); block_table int32 [B, max_blocks]: position j of
    sequence b is row j % block_size of block block_table[b, j // block_size]. Entries
    that are negative or out of range are never followed: the positions they cover
    become NaN rows, which a correct attention never reads (positions outside every
    window row's sliding window)."""
    k_pages = np.asarray(k_pages)
    v_pages = np.asarray(v_pages)
    nb, bs = k_pages.shape[0], k_pages.shape[1]
    table = np.asarray(block_table, dtype=np.int64)
    T = np.asarray(seq_lens, dtype=np.int64)
    R = T + np.asarray(draft_len, dtype=np.int64) + 1
    kflat = k_pages.reshape(nb * bs, Hkv, d)
    vflat = v_pages.reshape(nb * bs, Hkv, d)
    nan = 0x7F if k_pages.dtype == np.uint8 else 0x7FC0
    k = np.full((int(R.sum()), Hkv, d), nan, dtype=k_pages.dtype)
    v = np.full((int(R.sum()), Hkv, d), nan, dtype=v_pages.dtype)
    row0 = 0
    for b in range(len(T)):
        j = np.arange(int(R[b]))
        blk = table[b, j // bs]
        ok = (blk >= 0) & (blk < nb)
        src = blk[ok] * bs + j[ok] % bs
        k[row0 + j[ok]] = kflat[src]
        v[row0 + j[ok]] = vflat[src]
        row0 += int(R[b])
    return verify_attn(q, k, v, seq_lens, draft_len, Hq=Hq, Hkv=Hkv, d=d, kv_scale=kv_scale,
                       window=window, **kw)


def verify_attn_online(q, k, v, seq_lens, draft_len, *, tile, **kw):
    """The online-softmax (tile-by-tile) variant of ``verify_attn``."""
    return verify_attn(q, k, v, seq_lens, draft_len, online_tile=tile, **kw)


def argmax_rows(logits, nthreads=0):
    """logits: [rows, V] fp32, or uint16 bf16 bits. Returns int32 [rows]."""
    logits = np.ascontiguousarray(logits)
    if logits.dtype == np.uint16:
        dt = 0
    elif logits.dtype == np.float32:
        dt = 2
    else:
        raise TypeError("logits must be float32 or uint16 (bf16 bits)")
    rows, vocab = logits.shape
    amax = np.empty(rows, dtype=np.int32)
    if _load().orc_argmax_rows(rows, vocab, dt, _ptr(logits), _ptr(amax), int(nthreads)):
        raise ValueError("oracle rejected the arguments")
    return amax


def accept(amax, draft_tokens, draft_len):
    """First-mismatch acceptance from per-row argmax. Returns (accept_len, next_token)."""
    amax = np.ascontiguousarray(amax, dtype=np.int32)
    draft_tokens = np.ascontiguousarray(draft_tokens, dtype=np.int32)
    draft_len = np.ascontiguousarray(draft_len, dtype=np.int32)
    B = draft_len.shape[0]
    if amax.shape[0] != int(np.sum(draft_len.astype(np.int64) + 1)):
        raise ValueError("amax must have sum(1 + D_b) rows")
    if draft_tokens.shape[0] != int(np.sum(draft_len.astype(np.int64))):
        raise ValueError("draft_tokens must have sum(D_b) entries")
    al = np.empty(B, dtype=np.int32)
    nt = np.empty(B, dtype=np.int32)
    if _load().orc_accept(B, _ptr(draft_len), _ptr(draft_tokens), _ptr(amax), _ptr(al),
                          _ptr(nt)):
        raise ValueError("oracle rejected the arguments")
    return al, nt


def spec_accept(logits, draft_tokens, draft_len, nthreads=0):
    """Argmax of every window row, then first-mismatch acceptance."""
    amax = argmax_rows(logits, nthreads)
    al, nt = accept(amax, draft_tokens, draft_len)
    return al, nt, amax


def draft_signals(logits, nthreads=0):
    """logits: [rows, V] fp32, or uint16 bf16 bits. Returns (confidence, entropy), fp64
    [rows] each: the largest probability and the entropy in nats of each row's softmax."""
    logits = np.ascontiguousarray(logits)
    if logits.dtype == np.uint16:
        dt = 0
    elif logits.dtype == np.float32:
        dt = 2
    else:
        raise TypeError("logits must be float32 or uint16 (bf16 bits)")
    rows, vocab = logits.shape
    conf = np.empty(rows, dtype=np.float64)
    ent = np.empty(rows, dtype=np.float64)
    if _load().orc_draft_signals(rows, vocab, dt, _ptr(logits), _ptr(conf), _ptr(ent),
                                 int(nthreads)):
        raise ValueError("oracle rejected the arguments")
    return conf, ent


def accept_stochastic(target_logits, draft_logits, draft_tokens, draft_len, u_accept,
                      u_sample, temperature=1.0):
    """target_logits [sum (1 + D_b), V] and draft_logits [sum D_b, V], fp32 or uint16 bf16
    bits (the same type); draft_tokens int32 [sum D_b]; u_accept float32 [sum D_b] and
    u_sample float32 [B], uniform in [0, 1). Returns (accept_len, next_token,
    margin_accept, margin_sample): the acceptance length in [1, 1 + D_b], the emitted
    token, and per sequence the smallest relative margin of its keep / reject decisions and
    the relative margin of its draw (see oracle.c)."""
    t = np.ascontiguousarray(target_logits)
    dl = np.ascontiguousarray(draft_logits)
    if t.dtype != dl.dtype or t.dtype not in (np.uint16, np.float32):
        raise TypeError("logits must both be float32 or both uint16 (bf16 bits)")
    dt = 0 if t.dtype == np.uint16 else 2
    draft_len = np.ascontiguousarray(draft_len, dtype=np.int32)
    draft_tokens = np.ascontiguousarray(draft_tokens, dtype=np.int32)
    u_accept = np.ascontiguousarray(u_accept, dtype=np.float32)
    u_sample = np.ascontiguousarray(u_sample, dtype=np.float32)
    B = draft_len.shape[0]
    nd = int(np.sum(draft_len.astype(np.int64)))
    V = t.shape[1]
    if t.shape[0] != nd + B or (nd and dl.shape != (nd, V)) or draft_tokens.shape[0] != nd \
            or u_accept.shape[0] != nd or u_sample.shape[0] != B:
        raise ValueError("inconsistent shapes")
    if nd == 0:
        dl = np.zeros((1, V), dtype=t.dtype)
        draft_tokens = np.zeros(1, dtype=np.int32)
        u_accept = np.zeros(1, dtype=np.float32)
    al = np.empty(B, dtype=np.int32)
    nt = np.empty(B, dtype=np.int32)
    ma = np.empty(B, dtype=np.float64)
    ms = np.empty(B, dtype=np.float64)
    lib = _load()
    if lib.orc_accept_stochastic(B, V, dt, _ptr(t), _ptr(dl), _ptr(draft_tokens),
                                 _ptr(draft_len), _ptr(u_accept), _ptr(u_sample),
                                 ctypes.c_double(float(temperature)), _ptr(al), _ptr(nt),
                                 _ptr(ma), _ptr(ms)):
        raise ValueError("oracle rejected the arguments")
    return al, nt, ma, ms


def stochastic_decisions(target_logits, draft_logits, draft_tokens, draft_len, u_accept,
                         temperature=1.0):
    """Signed relative margin of every draft position's keep / reject decision
    (float64 [sum D_b]): (p(x) - u q(x)) / max(u q(x), p(x)), 0 when both are 0. Positive
    means kept; the acceptance length of ``accept_stochastic`` is 1 + the number of
    leading positive values of the sequence. Same arguments as ``accept_stochastic``
    without ``u_sample``."""
    t = np.ascontiguousarray(target_logits)
    dl = np.ascontiguousarray(draft_logits)
    if t.dtype != dl.dtype or t.dtype not in (np.uint16, np.float32):
        raise TypeError("logits must both be float32 or both uint16 (bf16 bits)")
    dt = 0 if t.dtype == np.uint16 else 2
    draft_len = np.ascontiguousarray(draft_len, dtype=np.int32)
    draft_tokens = np.ascontiguousarray(draft_tokens, dtype=np.int32)
    u_accept = np.ascontiguousarray(u_accept, dtype=np.float32)
    B = draft_len.shape[0]
    nd = int(np.sum(draft_len.astype(np.int64)))
    V = t.shape[1]
    if t.shape[0] != nd + B or (nd and dl.shape != (nd, V)) or draft_tokens.shape[0] != nd \
            or u_accept.shape[0] != nd:
        raise ValueError("inconsistent shapes")
    out = np.empty(max(nd, 1), dtype=np.float64)
    if nd == 0:
        return out[:0]
    if _load().orc_stochastic_decisions(B, V, dt, _ptr(t), _ptr(dl), _ptr(draft_tokens),
                                        _ptr(draft_len), _ptr(u_accept),
                                        ctypes.c_double(float(temperature)), _ptr(out)):
        raise ValueError("oracle rejected the arguments")
    return out
