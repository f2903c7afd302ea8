"""Shared helpers of the GPU parity tests: move generated inputs to the device, call the
C-ABI path, compare with the fp64 oracle."""
import numpy as np
import torch

import oracle
import speculative_decoding_verification_gqa_gb300 as sv
from speculative_decoding_verification_gqa_gb300 import build

ABS_TOL = 1e-2   # max |gpu - oracle| beyond the bf16 output rounding (see compare)
REL_TOL = 2e-2   # max |gpu - oracle| / max |oracle| (normwise)

_built = False


def ensure_built():
    global _built
    if not _built:
        build.build()
        sv.load_library()
        _built = True


def dev_attn(x, device="cuda"):
    q = torch.from_numpy(x["q"].view(np.int16)).view(torch.bfloat16).to(device)
    if x["k"].dtype == np.uint8:
        k = torch.from_numpy(x["k"]).to(device)
        v = torch.from_numpy(x["v"]).to(device)
        sc = torch.from_numpy(x["kv_scale"]).to(device)
    else:
        k = torch.from_numpy(x["k"].view(np.int16)).view(torch.bfloat16).to(device)
        v = torch.from_numpy(x["v"].view(np.int16)).view(torch.bfloat16).to(device)
        sc = None
    T = torch.from_numpy(x["seq_lens"].astype(np.int32)).to(device)
    D = torch.from_numpy(x["draft_len"].astype(np.int32)).to(device)
    return q, k, v, sc, T, D


def gpu_attn(x, *, max_draft=None, max_seq=None, workspace=None, out=None, window=0):
    q, k, v, sc, T, D = dev_attn(x)
    md = int(x["draft_len"].max()) if max_draft is None else max_draft
    ms = int(x["seq_lens"].max()) if max_seq is None else max_seq
    o = sv.spec_verify_attn(q, k, v, T, D, max_draft_len=md, max_seq_len=ms, kv_scale=sc,
                            workspace=workspace, out=out, sliding_window=window)
    torch.cuda.synchronize()
    return o.view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_to_f64(bits):
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def bf16_half_ulp(x):
    """Half the bf16 spacing at |x| (8 significant bits): the rounding error that storing
    an exact result in the bf16 output format can add by itself."""
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, np.exp2(e - 8), 0.0)


def compare(gpu_bits, ref, rows_mask=None, raw=False):
    """Returns (max_abs, normwise_rel) over the outputs where ref is finite. max_abs is the
    error beyond the bf16 output format's own rounding: max(|g - r| - half_ulp(max(|g|,
    |r|)), 0); normwise_rel = max |g - r| / max |r|. With raw=True a third value is the
    plain max |g - r|."""
    g = bf16_to_f64(gpu_bits)
    sel = np.isfinite(ref)
    if rows_mask is not None:
        sel &= rows_mask
    assert sel.any()
    assert np.isfinite(g[sel]).all(), "non-finite GPU output"
    err = np.abs(g[sel] - ref[sel])
    excess = np.maximum(err - bf16_half_ulp(np.maximum(np.abs(g[sel]), np.abs(ref[sel]))), 0.0)
    res = (float(excess.max()), float(err.max() / np.abs(ref[sel]).max()))
    return res + (float(err.max()),) if raw else res


def assert_close(gpu_bits, ref):
    """The parity bound: error beyond the output format's rounding <= ABS_TOL and normwise
    relative error <= REL_TOL. The plain max |gpu - oracle| and max |oracle| are reported
    beside them (printed, and in the assertion message)."""
    ma, mr, raw = compare(gpu_bits, ref, raw=True)
    peak = float(np.abs(ref[np.isfinite(ref)]).max())
    msg = ("max|gpu-oracle| beyond bf16 half-ulp %.3g (bound %g), plain max|gpu-oracle| %.3g, "
           "max|oracle| %.3g, normwise rel %.3g (bound %g)" % (ma, ABS_TOL, raw, peak, mr, REL_TOL))
    print(msg)
    assert ma <= ABS_TOL and mr <= REL_TOL, msg
    return ma, mr


def oracle_attn(w, x, units=None, window=0):
    return oracle.verify_attn(x["q"], x["k"], x["v"], x["seq_lens"], x["draft_len"], Hq=w.Hq,
                              Hkv=w.Hkv, d=w.d, kv_scale=x["kv_scale"], units=units,
                              window=window)


def dev_accept(a, device="cuda"):
    if a["logits"].dtype == np.uint16:
        lg = torch.from_numpy(a["logits"].view(np.int16)).view(torch.bfloat16).to(device)
    else:
        lg = torch.from_numpy(a["logits"]).to(device)
    dt = torch.from_numpy(a["draft_tokens"].astype(np.int32)).to(device)
    dl = torch.from_numpy(a["draft_len"].astype(np.int32)).to(device)
    return lg, dt, dl


def gpu_accept(a, max_draft=None):
    lg, dt, dl = dev_accept(a)
    md = int(a["draft_len"].max()) if max_draft is None else max_draft
    tgt = torch.full((lg.shape[0],), -1, dtype=torch.int32, device="cuda")
    al, nt = sv.spec_accept(lg, dt, dl, max_draft_len=md, target_tokens=tgt)
    torch.cuda.synchronize()
    return al.cpu().numpy(), nt.cpu().numpy(), tgt.cpu().numpy()
