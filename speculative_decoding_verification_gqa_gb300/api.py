"""Thin Python binding of libspecverify.so (ctypes). Argument marshalling only: every
step of the verification path runs in the library's CUDA kernels; there is no CPU or
PyTorch fallback, and every call raises if the library is missing or returns an error.

PyTorch supplies device memory and the current stream. Entry points mirror the C ABI in
include/specverify.h:

* ``spec_verify_attn`` -- GQA verify attention over cached prefix + draft window.
* ``spec_verify_attn_paged`` -- the same over a paged cache (block pool + block table).
* ``spec_verify_attn_host_lengths`` -- the same with host copies of the lengths (plan on
  the host, no planning kernel).
* ``spec_accept`` -- greedy acceptance (argmax per window row, first mismatch).
* ``spec_accept_stochastic`` -- distribution-preserving acceptance for sampled decoding.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libspecverify.so")

SV_BF16, SV_FP8_E4M3, SV_FP32 = 0, 1, 2
STATUS = {0: "SV_OK", 1: "SV_ERR_NULL", 2: "SV_ERR_SHAPE", 3: "SV_ERR_DTYPE",
          4: "SV_ERR_ALIGN", 5: "SV_ERR_WORKSPACE", 6: "SV_ERR_CUDA", 7: "SV_ERR_TIMEOUT",
          8: "SV_ERR_DEVICE_SHAPE"}
EXPORTS = ("spec_verify_attn_workspace_size", "spec_verify_attn", "spec_verify_attn_paged",
           "spec_verify_attn_host_lengths",
           "spec_accept_workspace_size",
           "spec_accept", "spec_draft_signals_workspace_size", "spec_draft_signals",
           "sv_workspace_status", "sv_status_string", "sv_set_attn_kernel", "sv_set_unit_ctas",
           "sv_set_profile_events", "sv_version", "sv_plan_preview",
           "sv_inject_launch_failure", "sv_inject_wait_timeout", "sv_set_row_pairs",
           "sv_row_pair_mode", "sv_set_kv_rings",
           "spec_accept_stochastic_workspace_size",
           "spec_accept_stochastic")


class SpecVerifyError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s failed: %s (%d)" % (where, STATUS.get(status, "?"), status))


class PlanInfo(ctypes.Structure):
    _fields_ = [("num_units", ctypes.c_int32), ("total_tiles", ctypes.c_int32),
                ("tile_keys", ctypes.c_int32), ("num_ctas", ctypes.c_int32),
                ("unit_ctas", ctypes.c_int32), ("switch_tiles", ctypes.c_int32)]


class AttnDesc(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("max_draft_len", ctypes.c_int32), ("max_seq_len", ctypes.c_int32),
                ("q_rows", ctypes.c_int64), ("kv_rows", ctypes.c_int64),
                ("kv_dtype", ctypes.c_int32), ("softmax_scale", ctypes.c_float),
                ("sliding_window", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libspecverify.so (built by ``build.build()``); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError("libspecverify.so is not built (%s); run "
                               "speculative_decoding_verification_gqa_gb300.build.build()" % path)
        lib = ctypes.CDLL(path)
        vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32
        lib.spec_verify_attn_workspace_size.argtypes = [ctypes.POINTER(AttnDesc)]
        lib.spec_verify_attn_workspace_size.restype = sz
        lib.spec_verify_attn.argtypes = [ctypes.POINTER(AttnDesc), vp, vp, vp, vp, vp, vp, vp,
                                         vp, sz, vp]
        lib.spec_verify_attn.restype = ctypes.c_int
        i64 = ctypes.c_int64
        lib.spec_verify_attn_paged.argtypes = [ctypes.POINTER(AttnDesc), vp, vp, vp, i64, i32,
                                               vp, i32, vp, vp, vp, vp, vp, sz, vp]
        lib.spec_verify_attn_paged.restype = ctypes.c_int
        lib.spec_verify_attn_host_lengths.argtypes = [ctypes.POINTER(AttnDesc), vp, vp, vp, vp,
                                                      vp, vp, vp, vp, vp, vp, sz, vp]
        lib.spec_verify_attn_host_lengths.restype = ctypes.c_int
        lib.spec_accept_workspace_size.argtypes = [i32, i32, i32]
        lib.spec_accept_workspace_size.restype = sz
        lib.spec_accept.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        lib.spec_accept.restype = ctypes.c_int
        lib.spec_draft_signals_workspace_size.argtypes = [i32, i32]
        lib.spec_draft_signals_workspace_size.restype = sz
        lib.spec_draft_signals.argtypes = [i32, i32, i32, vp, vp, vp, vp, sz, vp]
        lib.spec_draft_signals.restype = ctypes.c_int
        lib.sv_workspace_status.argtypes = [vp, ctypes.c_int, vp]
        lib.sv_workspace_status.restype = ctypes.c_int
        lib.sv_status_string.argtypes = [ctypes.c_int]
        lib.sv_status_string.restype = ctypes.c_char_p
        lib.sv_set_attn_kernel.argtypes = [ctypes.c_int]
        lib.sv_set_attn_kernel.restype = ctypes.c_int
        lib.sv_set_unit_ctas.argtypes = [ctypes.c_int]
        lib.sv_set_unit_ctas.restype = ctypes.c_int
        lib.sv_set_profile_events.argtypes = [vp, vp]
        lib.sv_set_profile_events.restype = None
        lib.sv_version.restype = ctypes.c_int
        lib.sv_plan_preview.argtypes = [ctypes.POINTER(AttnDesc), i32, vp, vp, i32, i32,
                                        ctypes.POINTER(PlanInfo), vp, vp, vp, i32]
        lib.sv_plan_preview.restype = ctypes.c_int
        lib.spec_accept_stochastic_workspace_size.argtypes = [i32, i32, i32]
        lib.spec_accept_stochastic_workspace_size.restype = sz
        lib.spec_accept_stochastic.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp, vp, vp,
                                               ctypes.c_float, vp, vp, vp, sz, vp]
        lib.spec_accept_stochastic.restype = ctypes.c_int
        lib.sv_inject_launch_failure.argtypes = [ctypes.c_int]
        lib.sv_inject_launch_failure.restype = ctypes.c_int
        lib.sv_inject_wait_timeout.argtypes = [ctypes.c_int64]
        lib.sv_inject_wait_timeout.restype = ctypes.c_int
        lib.sv_set_row_pairs.argtypes = [ctypes.c_int]
        lib.sv_set_row_pairs.restype = ctypes.c_int
        lib.sv_set_kv_rings.argtypes = [ctypes.c_int]
        lib.sv_set_kv_rings.restype = ctypes.c_int
        lib.sv_row_pair_mode.argtypes = [ctypes.POINTER(AttnDesc), i32, i32, i32]
        lib.sv_row_pair_mode.restype = ctypes.c_int
        _lib = lib
        return lib


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _or_placeholder(t: torch.Tensor) -> torch.Tensor:
    """t, or a small allocation of its dtype on its device when t is empty (a batch without
    drafts: the library requires the pointer when max_draft_len > 0 but never reads it)."""
    return t if t.numel() > 0 else torch.empty(16, dtype=t.dtype, device=t.device)


def _check(st: int, where: str):
    if st != 0:
        raise SpecVerifyError(st, where)


def _need(t: torch.Tensor, name: str, dtypes):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if t.dtype not in dtypes:
        raise TypeError("%s has dtype %s, expected one of %s" % (name, t.dtype, dtypes))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def attn_desc(q: torch.Tensor, k_cache: torch.Tensor, batch: int, max_draft_len: int,
              max_seq_len: int, softmax_scale: float = 0.0, sliding_window: int = 0) -> AttnDesc:
    fp8 = k_cache.dtype in (torch.uint8, torch.float8_e4m3fn)
    return AttnDesc(batch=batch, num_q_heads=q.shape[1], num_kv_heads=k_cache.shape[1],
                    head_dim=q.shape[2], max_draft_len=max_draft_len, max_seq_len=max_seq_len,
                    q_rows=q.shape[0], kv_rows=k_cache.shape[0],
                    kv_dtype=SV_FP8_E4M3 if fp8 else SV_BF16,
                    softmax_scale=float(softmax_scale), sliding_window=int(sliding_window))


def verify_workspace_bytes(desc: AttnDesc) -> int:
    n = load_library().spec_verify_attn_workspace_size(ctypes.byref(desc))
    if n == 0:
        raise SpecVerifyError(2, "spec_verify_attn_workspace_size")
    return n


def accept_workspace_bytes(batch: int, max_draft_len: int, vocab: int) -> int:
    n = load_library().spec_accept_workspace_size(batch, max_draft_len, vocab)
    if n == 0:
        raise SpecVerifyError(2, "spec_accept_workspace_size")
    return n


def signals_workspace_bytes(rows: int, vocab: int) -> int:
    n = load_library().spec_draft_signals_workspace_size(rows, vocab)
    if n == 0:
        raise SpecVerifyError(2, "spec_draft_signals_workspace_size")
    return n


def new_workspace(nbytes: int, device=None) -> torch.Tensor:
    """A zero-filled device workspace (the library's flag word must start at zero)."""
    return torch.zeros(nbytes, dtype=torch.uint8, device=device or "cuda")


def spec_verify_attn(q, k_cache, v_cache, seq_lens, draft_len, *, max_draft_len: int,
                     max_seq_len: int, kv_scale=None, out=None, workspace=None,
                     softmax_scale: float = 0.0, sliding_window: int = 0,
                     stream=None) -> torch.Tensor:
    """q [rows, Hq, d] bf16; k_cache/v_cache [kv_rows, Hkv, d] bf16, or uint8 /
    float8_e4m3fn E4M3 codes with kv_scale fp32 [2, Hkv]; seq_lens, draft_len int32 [B].
    Returns out [rows, Hq, d] bf16 (only the packed rows sum_b (1 + D_b) are written).
    ``sliding_window`` = W >= 1 restricts window row i to keys max(0, T+i-W+1) .. T+i."""
    _need(q, "q", (torch.bfloat16,))
    _need(k_cache, "k_cache", (torch.bfloat16, torch.uint8, torch.float8_e4m3fn))
    _need(v_cache, "v_cache", (k_cache.dtype,))
    _need(seq_lens, "seq_lens", (torch.int32,))
    _need(draft_len, "draft_len", (torch.int32,))
    if kv_scale is not None:
        _need(kv_scale, "kv_scale", (torch.float32,))
    if q.dim() != 3 or k_cache.dim() != 3 or v_cache.shape != k_cache.shape:
        raise ValueError("q must be [rows, Hq, d], k/v caches [kv_rows, Hkv, d]")
    desc = attn_desc(q, k_cache, seq_lens.shape[0], max_draft_len, max_seq_len, softmax_scale,
                     sliding_window)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", (torch.bfloat16,))
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    if workspace is None:
        workspace = new_workspace(verify_workspace_bytes(desc), q.device)
    st = load_library().spec_verify_attn(
        ctypes.byref(desc), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seq_lens),
        _ptr(draft_len), _ptr(kv_scale), _ptr(out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "spec_verify_attn")
    return out


def spec_verify_attn_host_lengths(q, k_cache, v_cache, seq_lens, draft_len, seq_lens_host,
                                  draft_len_host, *, max_draft_len: int, max_seq_len: int,
                                  kv_scale=None, out=None, workspace=None,
                                  softmax_scale: float = 0.0, sliding_window: int = 0,
                                  stream=None) -> torch.Tensor:
    """spec_verify_attn with the lengths also in host memory (int32 CPU tensors equal to
    seq_lens and draft_len): the work plan is made on the host and travels with the
    attention launch."""
    for t, n in ((seq_lens_host, "seq_lens_host"), (draft_len_host, "draft_len_host")):
        if t.device.type != "cpu" or t.dtype != torch.int32 or not t.is_contiguous():
            raise ValueError("%s must be a contiguous int32 CPU tensor" % n)
    _need(q, "q", (torch.bfloat16,))
    _need(k_cache, "k_cache", (torch.bfloat16, torch.uint8, torch.float8_e4m3fn))
    _need(v_cache, "v_cache", (k_cache.dtype,))
    _need(seq_lens, "seq_lens", (torch.int32,))
    _need(draft_len, "draft_len", (torch.int32,))
    if kv_scale is not None:
        _need(kv_scale, "kv_scale", (torch.float32,))
    if q.dim() != 3 or k_cache.dim() != 3 or v_cache.shape != k_cache.shape:
        raise ValueError("q must be [rows, Hq, d], k/v caches [kv_rows, Hkv, d]")
    if seq_lens_host.numel() != seq_lens.numel() or draft_len_host.numel() != draft_len.numel():
        raise ValueError("host and device length arrays differ in size")
    desc = attn_desc(q, k_cache, seq_lens.shape[0], max_draft_len, max_seq_len, softmax_scale,
                     sliding_window)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", (torch.bfloat16,))
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    if workspace is None:
        workspace = new_workspace(verify_workspace_bytes(desc), q.device)
    st = load_library().spec_verify_attn_host_lengths(
        ctypes.byref(desc), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seq_lens),
        _ptr(draft_len), ctypes.c_void_p(seq_lens_host.data_ptr()),
        ctypes.c_void_p(draft_len_host.data_ptr()), _ptr(kv_scale), _ptr(out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "spec_verify_attn_host_lengths")
    return out


def spec_verify_attn_paged(q, k_pages, v_pages, block_table, seq_lens, draft_len, *,
                           max_draft_len: int, max_seq_len: int, kv_scale=None, out=None,
                           workspace=None, softmax_scale: float = 0.0, sliding_window: int = 0,
                           stream=None) -> torch.Tensor:
    """spec_verify_attn over a paged cache. k_pages/v_pages [num_blocks, block_size, Hkv, d]
    (bf16, or uint8 / float8_e4m3fn codes with kv_scale); block_table int32 [B, max_blocks]:
    position j of sequence b is row j % block_size of block block_table[b, j // block_size]."""
    _need(q, "q", (torch.bfloat16,))
    _need(k_pages, "k_pages", (torch.bfloat16, torch.uint8, torch.float8_e4m3fn))
    _need(v_pages, "v_pages", (k_pages.dtype,))
    _need(block_table, "block_table", (torch.int32,))
    _need(seq_lens, "seq_lens", (torch.int32,))
    _need(draft_len, "draft_len", (torch.int32,))
    if kv_scale is not None:
        _need(kv_scale, "kv_scale", (torch.float32,))
    if q.dim() != 3 or k_pages.dim() != 4 or v_pages.shape != k_pages.shape:
        raise ValueError("q must be [rows, Hq, d], k/v pages [num_blocks, block_size, Hkv, d]")
    if block_table.dim() != 2 or block_table.shape[0] != seq_lens.shape[0]:
        raise ValueError("block_table must be [B, max_blocks]")
    nb, bs = k_pages.shape[0], k_pages.shape[1]
    flat = k_pages.view(nb * bs, k_pages.shape[2], k_pages.shape[3])
    desc = attn_desc(q, flat, seq_lens.shape[0], max_draft_len, max_seq_len, softmax_scale,
                     sliding_window)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", (torch.bfloat16,))
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    if workspace is None:
        workspace = new_workspace(verify_workspace_bytes(desc), q.device)
    st = load_library().spec_verify_attn_paged(
        ctypes.byref(desc), _ptr(q), _ptr(k_pages), _ptr(v_pages), nb, bs, _ptr(block_table),
        block_table.shape[1], _ptr(seq_lens), _ptr(draft_len), _ptr(kv_scale), _ptr(out),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "spec_verify_attn_paged")
    return out


def spec_accept(logits, draft_tokens, draft_len, *, max_draft_len: int, accept_len=None,
                next_token=None, target_tokens=None, workspace=None, stream=None):
    """logits [sum (1 + D_b), V] bf16 or fp32; draft_tokens int32 [sum D_b]; draft_len int32
    [B]. Returns (accept_len, next_token), int32 [B] each; fills ``target_tokens`` (int32
    [sum (1 + D_b)]) with the target's greedy token per row when it is given."""
    _need(logits, "logits", (torch.bfloat16, torch.float32))
    _need(draft_tokens, "draft_tokens", (torch.int32,))
    _need(draft_len, "draft_len", (torch.int32,))
    B = draft_len.shape[0]
    V = logits.shape[-1]
    if accept_len is None:
        accept_len = torch.empty(B, dtype=torch.int32, device=logits.device)
    if next_token is None:
        next_token = torch.empty(B, dtype=torch.int32, device=logits.device)
    for t, n in ((accept_len, "accept_len"), (next_token, "next_token")):
        _need(t, n, (torch.int32,))
    if target_tokens is not None:
        _need(target_tokens, "target_tokens", (torch.int32,))
    if workspace is None:
        workspace = new_workspace(accept_workspace_bytes(B, max_draft_len, V), logits.device)
    dt = SV_BF16 if logits.dtype == torch.bfloat16 else SV_FP32
    dtok = _or_placeholder(draft_tokens)
    st = load_library().spec_accept(
        B, max_draft_len, V, dt, _ptr(logits), _ptr(dtok), _ptr(draft_len), _ptr(accept_len),
        _ptr(next_token), _ptr(target_tokens), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "spec_accept")
    return accept_len, next_token


def spec_accept_stochastic(target_logits, draft_logits, draft_tokens, draft_len, u_accept,
                           u_sample, *, max_draft_len: int, temperature: float = 1.0,
                           accept_len=None, next_token=None, workspace=None, stream=None):
    """Distribution-preserving acceptance for sampled decoding. target_logits [sum (1 + D_b),
    V] and draft_logits [sum D_b, V] (bf16 or fp32, the same); draft_tokens int32 [sum
    D_b]; draft_len int32 [B]; u_accept fp32 [sum D_b] and u_sample fp32 [B], uniform in
    [0, 1). Returns (accept_len, next_token), int32 [B] each."""
    _need(target_logits, "target_logits", (torch.bfloat16, torch.float32))
    _need(draft_logits, "draft_logits", (target_logits.dtype,))
    _need(draft_tokens, "draft_tokens", (torch.int32,))
    _need(draft_len, "draft_len", (torch.int32,))
    _need(u_accept, "u_accept", (torch.float32,))
    _need(u_sample, "u_sample", (torch.float32,))
    B = draft_len.shape[0]
    V = target_logits.shape[-1]
    if draft_logits.dim() != 2 or draft_logits.shape[1] != V:
        raise ValueError("draft_logits must be [sum D_b, V] with the target's V")
    if u_sample.numel() != B:
        raise ValueError("u_sample must hold one draw per sequence")
    if accept_len is None:
        accept_len = torch.empty(B, dtype=torch.int32, device=target_logits.device)
    if next_token is None:
        next_token = torch.empty(B, dtype=torch.int32, device=target_logits.device)
    for t, n in ((accept_len, "accept_len"), (next_token, "next_token")):
        _need(t, n, (torch.int32,))
    lib = load_library()
    if workspace is None:
        n = lib.spec_accept_stochastic_workspace_size(B, max_draft_len, V)
        if n == 0:
            raise SpecVerifyError(2, "spec_accept_stochastic_workspace_size")
        workspace = new_workspace(n, target_logits.device)
    dt = SV_BF16 if target_logits.dtype == torch.bfloat16 else SV_FP32
    dlg, dtk, ua = (_or_placeholder(t) for t in (draft_logits, draft_tokens, u_accept))
    st = lib.spec_accept_stochastic(
        B, max_draft_len, V, dt, _ptr(target_logits), _ptr(dlg), _ptr(dtk), _ptr(draft_len),
        _ptr(ua),
        _ptr(u_sample), float(temperature), _ptr(accept_len), _ptr(next_token),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "spec_accept_stochastic")
    return accept_len, next_token


def spec_draft_signals(logits, *, confidence=None, entropy=None, workspace=None, stream=None):
    """logits [rows, V] bf16 or fp32 (e.g. the draft model's logits at each drafted
    position). Returns (confidence, entropy), fp32 [rows] each: the largest probability
    and the entropy (nats) of each row's softmax."""
    _need(logits, "logits", (torch.bfloat16, torch.float32))
    rows, V = logits.shape
    if confidence is None:
        confidence = torch.empty(rows, dtype=torch.float32, device=logits.device)
    if entropy is None:
        entropy = torch.empty(rows, dtype=torch.float32, device=logits.device)
    for t, n in ((confidence, "confidence"), (entropy, "entropy")):
        _need(t, n, (torch.float32,))
    if workspace is None:
        workspace = new_workspace(signals_workspace_bytes(rows, V), logits.device)
    dt = SV_BF16 if logits.dtype == torch.bfloat16 else SV_FP32
    st = load_library().spec_draft_signals(
        rows, V, dt, _ptr(logits), _ptr(confidence), _ptr(entropy), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "spec_draft_signals")
    return confidence, entropy


def workspace_status(workspace: torch.Tensor, clear: bool = False, stream=None) -> int:
    """Synchronises and returns the workspace's sticky device-side status (0 = ok)."""
    return load_library().sv_workspace_status(_ptr(workspace), int(clear), _stream(stream))


def set_attn_kernel(which: int) -> int:
    """0 automatic, 1 mma.sync kernel, 2 tcgen05 kernel. Returns the previous choice."""
    prev = load_library().sv_set_attn_kernel(int(which))
    if prev < 0:
        raise ValueError("attention kernel %d is not available" % which)
    return prev


def set_unit_ctas(mode: int) -> int:
    """-1 cost model (default), 0 split tile line, k >= 1 k CTAs per unit. Returns the
    previous mode."""
    prev = load_library().sv_set_unit_ctas(int(mode))
    if prev < -1:
        raise ValueError("unit-CTA mode must be in [-1, 1024]")
    return prev


def inject_launch_failure(after: int) -> int:
    """Test hook: after ``after`` more kernel launches of the library, the next one fails
    on the host, and the call that makes it raises SpecVerifyError (SV_ERR_CUDA); a
    negative ``after`` disarms. Returns the launches that were still to go before a
    pending failure, or -1."""
    return load_library().sv_inject_launch_failure(int(after))


def set_row_pairs(mode: int) -> int:
    """0 never (default), 1 whenever the row-pair kernel applies (128 < G(1 + max_draft) <=
    256, bf16, d = 128, packed, no window, B * Hkv <= SMs). Returns the previous mode."""
    prev = load_library().sv_set_row_pairs(int(mode))
    if prev < 0:
        raise ValueError("row-pair mode must be 0 or 1")
    return prev


def set_kv_rings(mode: int) -> int:
    """bf16 K/V on the tcgen05 kernel: -1 by the call's shape (default), 0 paired K + V
    stages, 1 separate K and V rings. Returns the previous mode."""
    prev = load_library().sv_set_kv_rings(int(mode))
    if prev < -1:
        raise ValueError("ring mode must be -1, 0 or 1")
    return prev


def row_pair_mode(desc, num_sms: int, attn_kernel: int = 2, block_size: int = 0) -> int:
    """1 if a call with this descriptor runs the row-pair kernel, else 0."""
    r = load_library().sv_row_pair_mode(ctypes.byref(desc), int(block_size), int(num_sms),
                                        int(attn_kernel))
    if r < 0:
        raise SpecVerifyError(2, "sv_row_pair_mode")
    return r


def inject_wait_timeout(limit_cycles: int) -> int:
    """Test hook: the next launch of the tcgen05 attention kernel waits at most
    ``limit_cycles`` clock cycles per barrier and each CTA withholds its first tile's
    loads, so the kernel gives up, sets SV_ERR_TIMEOUT in the workspace and returns. 0
    disarms.
    Returns 1 if an arming was pending, else 0."""
    return load_library().sv_inject_wait_timeout(int(limit_cycles))


def set_profile_events(start=None, stop=None):
    """Record CUDA events around the main attention kernel of later calls (None: off)."""
    lib = load_library()
    if start is None or stop is None:
        lib.sv_set_profile_events(None, None)
    else:
        lib.sv_set_profile_events(ctypes.c_void_p(start.cuda_event),
                                  ctypes.c_void_p(stop.cuda_event))


def plan_preview(desc: AttnDesc, seq_lens, draft_len, *, num_sms: int, attn_kernel: int = 2,
                 block_size: int = 0) -> dict:
    """The work plan a verify-attention call with these host lengths (int sequences) makes
    on a device of ``num_sms`` SMs, computed on the host by the library. Returns a dict:
    the sv_plan_info counts, ``units`` int32 [U, 4] (b, KV head, row tile, first cache
    position of the unit's first tile), ``unit_begin`` int32 [U + 1] and ``cta_begin``
    int32 [C + 1, 2] (first tile, its unit)."""
    import numpy as np
    T = np.ascontiguousarray(seq_lens, dtype=np.int32)
    D = np.ascontiguousarray(draft_len, dtype=np.int32)
    if T.shape != (desc.batch,) or D.shape != (desc.batch,):
        raise ValueError("seq_lens and draft_len must hold desc.batch lengths")
    lib = load_library()
    info = PlanInfo()
    st = lib.sv_plan_preview(ctypes.byref(desc), block_size, T.ctypes.data, D.ctypes.data,
                             num_sms, attn_kernel, ctypes.byref(info), None, None, None, 0)
    _check(st, "sv_plan_preview")
    U, C = info.num_units, info.num_ctas
    units = np.zeros((max(U, 1), 4), dtype=np.int32)
    ubeg = np.zeros(U + 1, dtype=np.int32)
    cta = np.zeros((C + 1, 2), dtype=np.int32)
    st = lib.sv_plan_preview(ctypes.byref(desc), block_size, T.ctypes.data, D.ctypes.data,
                             num_sms, attn_kernel, ctypes.byref(info), units.ctypes.data,
                             ubeg.ctypes.data, cta.ctypes.data, U)
    _check(st, "sv_plan_preview")
    out = {name: getattr(info, name) for name, _ in PlanInfo._fields_}
    out.update(units=units[:U], unit_begin=ubeg, cta_begin=cta)
    return out


def default_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)
