"""Benchmark of the verification step: verify attention + greedy acceptance.

One step = spec_verify_attn (plan, attention, split combine) + spec_accept (argmax,
first-mismatch scan) over one batch of seeded synthetic inputs already resident in HBM.
Default workload: the Llama-3-8B-shaped layer (B=16, Hq=32, Hkv=8, d=128, D=31,
T=8192, bf16 KV; logits [16, 32, 128256] bf16, draft match probability 0.8).

Prints one JSON line (rank 0). ``value`` is KV GB/s: algorithmic K/V bytes of all ranks
per step / the step time (max over ranks). ``--impl reference`` times the fp64 CPU oracle
on the host cores instead (a bounded sample of the same workload per step).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--config c2] [--D d] [--kernel auto|mma|tcgen05] [--no-e2e]
                       [--no-cpu-baseline]
"""
from __future__ import annotations

import argparse
import json
import os
import shutil
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "spec-verify attention: KV GB/s vs HBM peak; accepted tokens/s"


# ---------------------------------------------------------------- ranks (replicas only)
# One process per GPU under torchrun. Each rank verifies its own batch (no data-path
# collective); the only exchange is the max of the timings over ranks.

def rank_info():
    """(world size, rank, local rank) from the torchrun environment (1, 0, 0 without)."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def replica_seed(seed: int, rank: int) -> int:
    """Input seed of a rank: every replica verifies a different batch."""
    return seed + 7919 * rank


def max_over_ranks(values, device=None):
    """Element-wise maximum of `values` over all ranks of the default process group (the
    values themselves without one). NCCL reduces on `device`, gloo on the host."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    dev = device if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_rate(world: int, units_per_rank: float, seconds: float) -> float:
    """Units of all ranks per second of the slowest rank (weak scaling)."""
    return world * units_per_rank / seconds
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_BYTES = 129e6


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="c2", choices=["c1", "c2", "c3", "c4", "c5"])
    ap.add_argument("--D", type=int, default=None, help="draft length override (c4 sweep)")
    ap.add_argument("--kernel", default="auto", choices=["auto", "mma", "tcgen05"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--side-window", type=int, default=4096,
                    help="also time the verify call with this sliding window (0: skip)")
    ap.add_argument("--side-block", type=int, default=16,
                    help="also time the verify call over a paged copy of the cache with "
                         "blocks of this many positions (0: skip)")
    ap.add_argument("--side-stochastic", type=int, default=1,
                    help="also time spec_accept_stochastic on the step's shapes (0: skip)")
    ap.add_argument("--per-config", default="c3,c4:15,c4:16,c4:31,c4:31:pairs,c5",
                    help="other workloads measured into the line's per_config object, as "
                         "config[:D[:pairs]] items ('none': skip; only with the default "
                         "--config; ':pairs' runs the row-pair kernel)")
    ap.add_argument("--per-config-steps", type=int, default=100)
    ap.add_argument("--only-step", action="store_true",
                    help="run W + K steps of the workload and exit (for profilers)")
    ap.add_argument("--row-pairs", type=int, default=0, choices=[0, 1],
                    help="1: the row-pair attention kernel wherever it applies")
    ap.add_argument("--kv-rings", type=int, default=-1, choices=[-1, 0, 1],
                    help="bf16 K/V on the tcgen05 kernel: -1 by the call's shape (default), "
                         "0 paired K + V stages, 1 separate K and V rings")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def workload(args):
    from speculative_decoding_verification_gqa_gb300 import synth
    w = synth.CONFIGS[args.config]
    T, D, p = synth.lengths(w, args.seed, D=args.D)
    return w, T, D, p


def describe(w, T, D):
    G = w.G
    if w.ragged:
        shape = ("B=%d Hq=%d Hkv=%d d=%d T_b~U[%d,%d] D_b in %s (seed: sum T=%d, sum W=%d)"
                 % (w.B, w.Hq, w.Hkv, w.d, w.T_range[0], w.T_range[1], list(w.D_choices),
                    int(T.sum()), int((D + 1).sum())))
    else:
        shape = ("B=%d Hq=%d Hkv=%d (G=%d) d=%d D=%d (M=G*(1+D)=%d) T=%d"
                 % (w.B, w.Hq, w.Hkv, G, w.d, int(D[0]), G * (int(D[0]) + 1), int(T[0])))
    return "%s: %s, %s KV, logits V=%d %s" % (w.name, shape, w.kv_dtype, w.V, w.logits_dtype)


def algorithmic_bytes(w, T, D, window=0):
    """K+V bytes actually required (each KV element read once) and Q+out bytes. With a
    sliding window of W positions a sequence needs only positions max(0, T-W+1) .. T+D."""
    kv_elem = 1 if w.kv_dtype == "fp8_e4m3" else 2
    W = D.astype(np.int64) + 1
    rows = T.astype(np.int64) + W
    if window > 0:
        rows = rows - np.maximum(T.astype(np.int64) - window + 1, 0)
    kv = int(2 * w.Hkv * w.d * kv_elem * np.sum(rows))
    qo = int(2 * np.sum(W) * w.Hq * w.d * 2)
    return kv, qo


def flops(w, T, D):
    W = D.astype(np.int64) + 1
    # QK and PV over the visible keys of every row (window-causal): 4 * d per (row, key)
    keys = np.sum(W * T + W * (W + 1) // 2)
    return int(4 * w.Hq * w.d * keys)


# Nominal dense tensor rates of the part (PFLOP/s): e4m3 4.5, bf16/f16 2.25. Only bf16 is
# measured, so an e4m3 contraction's peak is the measured bf16 peak times their ratio.
E4M3_OVER_BF16 = 4.5 / 2.25


def tensor_seconds(fl, kv_dtype, attn_kernel, bf16_tflops):
    """Tensor-core time of the attention's algorithmic FLOPs at the peak of the type each
    contraction runs in. Q K^T and P V are half of the FLOPs each. bf16 K/V: both on the
    16-bit path. FP8 K/V on the tcgen05 kernel: Q K^T on the 8-bit path (E4M3 K, Q as E4M3
    terms) at the e4m3 peak, P V on the 16-bit path; on the mma.sync kernel both run in f16
    (K and V decoded)."""
    p16 = bf16_tflops * 1e12
    if kv_dtype == "fp8_e4m3" and attn_kernel == "tcgen05":
        return fl / 2.0 / (p16 * E4M3_OVER_BF16) + fl / 2.0 / p16
    return fl / p16


def roofline_record(kv_bytes, qo_bytes, fl, attn_s, hbm_gbs, bf16_tflops, kv_dtype,
                    attn_kernel, traffic=None):
    """The attention kernel against its roofline: the bound is the slower of its
    algorithmic bytes at the HBM peak and its algorithmic FLOPs at the tensor peak of their
    types; achieved and peak are in that bound's unit, frac = achieved / peak (the bound's
    time over the kernel's)."""
    nbytes = kv_bytes + qo_bytes
    t_hbm = nbytes / (hbm_gbs * 1e9)
    t_tc = tensor_seconds(fl, kv_dtype, attn_kernel, bf16_tflops)
    if t_hbm >= t_tc:
        bound, unit = "hbm", "GB/s"
        achieved, peak = nbytes / attn_s / 1e9, hbm_gbs
    else:
        bound, unit = "tensor", "TFLOP/s"
        achieved, peak = fl / attn_s / 1e12, fl / t_tc / 1e12
    return {"bound": bound, "achieved": round(achieved, 1), "peak": round(peak, 1),
            "unit": unit, "frac": round(achieved / peak, 4), "traffic": traffic,
            "algorithmic_bytes": nbytes, "algorithmic_flops": int(fl),
            "t_hbm_us": round(t_hbm * 1e6, 2), "t_tensor_us": round(t_tc * 1e6, 2)}


# The sources that define the verify-attention kernel's code and its work plan.
ATTN_SOURCES = ("attn_tc.cu", "tc_util.cuh", "internal.cuh", "plan_combine.cu", "api.cu")


def code_text(src: str) -> str:
    """C/C++/CUDA source without its comments and with whitespace runs collapsed to one
    space (string and character literals, such as inline PTX, are kept as written)."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":  # a literal: copy up to its unescaped closing quote
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash():
    """First 16 hex digits of the sha256 of the verify-attention kernel's sources and the
    library header, comments and layout left out: names the kernel version an ncu capture
    was taken of (edits to comments keep a capture valid)."""
    import hashlib
    pkg = os.path.join(ROOT, "speculative_decoding_verification_gqa_gb300", "csrc")
    files = [os.path.join(pkg, f) for f in ATTN_SOURCES]
    files.append(os.path.join(ROOT, "include", "specverify.h"))
    h = hashlib.sha256()
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, encoding="utf-8") as fh:
            h.update(code_text(fh.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(config, D, attn_kernel, src_hash=None):
    """DRAM bytes (read + written) per launch of the attention kernel from the ncu capture
    of this workload, or None when there is none for the current sources."""
    e = NCU_TRAFFIC.get((config, D, attn_kernel))
    if e is None:
        return None
    h, nbytes = e
    return nbytes if h == (src_hash or kernel_source_hash()) else None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        exe = shutil.which("nvidia-smi")
        if not exe:
            return
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        self.fh = open(self.path, "w")
        self.proc = subprocess.Popen([exe, "-i", str(self.index), "--query-gpu=" + self.Q,
                                      "--format=csv,noheader,nounits", "-lms", "50"],
                                     stdout=self.fh, stderr=subprocess.DEVNULL)
        time.sleep(0.3)

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [s.strip() for s in line.split(",")]
                if len(parts) >= 8:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4)
                          if r[4 + k].lower() == "active"})
        loaded = [s for s in sm if mx and s > 0.5 * max(mx)] or sm
        return {"sm_mhz": float(np.median(loaded)) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def row_keys(w, T, D):
    """Keys seen by every (packed window row, head) output, flattened [sum W * Hq]."""
    ks = [np.repeat(np.arange(Tb + 1, Tb + Db + 2, dtype=np.int64), w.Hq)
          for Tb, Db in zip(T.tolist(), D.tolist())]
    return np.concatenate(ks)


def cpu_oracle_sample(w, x, a, budget_s, seed, acc_rows=None):
    """Times the fp64 oracle on a random sample of the workload's output rows (attention)
    and on whole sequences' acceptance, then extrapolates to one whole step:
    t_step = t_attn_sample / f_attn + t_accept_sample / f_accept, where f is the fraction
    of the work sampled (attention: keys visited; acceptance: logit rows)."""
    import oracle
    rng = np.random.default_rng(seed + 99)
    T, D = x["seq_lens"], x["draft_len"]
    keys = row_keys(w, T, D)
    total_keys = float(keys.sum())
    order = rng.permutation(keys.size)
    done = 0
    t_attn = 0.0
    keys_done = 0.0
    target_keys = None
    threads = oracle.num_threads()
    while done < order.size:
        if target_keys is None:
            n = min(order.size - done, 2 * threads)
            pick = order[done:done + n]
        else:
            cum = np.cumsum(keys[order[done:]])
            n = int(np.searchsorted(cum, target_keys)) + 1
            pick = order[done:done + n]
        sel = np.zeros(keys.size, dtype=np.uint8)
        sel[pick] = 1
        t0 = time.perf_counter()
        oracle.verify_attn(x["q"], x["k"], x["v"], T, D, Hq=w.Hq, Hkv=w.Hkv, d=w.d,
                           kv_scale=x["kv_scale"], rows=sel)
        t_attn += time.perf_counter() - t0
        keys_done += float(keys[pick].sum())
        done += pick.size
        rate = keys_done / t_attn
        left = budget_s * 0.85 - t_attn
        if left <= 0.02 * budget_s:
            break
        target_keys = rate * left
    # acceptance: whole sequences, in random order, until ~15% of the budget
    W = D.astype(np.int64) + 1
    q_off = np.concatenate([[0], np.cumsum(W)])
    d_off = np.concatenate([[0], np.cumsum(D.astype(np.int64))])
    t_acc = 0.0
    rows_acc = 0
    accepted = 0
    for b in rng.permutation(len(D)):
        lg = a["logits"][q_off[b]:q_off[b + 1]]
        t0 = time.perf_counter()
        al, _, _ = oracle.spec_accept(lg, a["draft_tokens"][d_off[b]:d_off[b + 1]], D[b:b + 1])
        t_acc += time.perf_counter() - t0
        rows_acc += int(W[b])
        accepted += int(al[0])
        if t_acc >= budget_s * 0.15 or (acc_rows and rows_acc >= acc_rows):
            break
    f_attn = keys_done / total_keys
    f_acc = rows_acc / float(W.sum())
    t_step = t_attn / f_attn + t_acc / f_acc
    kv_bytes, _ = algorithmic_bytes(w, T, D)
    return dict(t_step=t_step, seconds=t_attn + t_acc, f_attn=f_attn, f_acc=f_acc,
                gbs=kv_bytes / t_step / 1e9, acc_per_s=accepted / f_acc / t_step,
                threads=threads, rows=int(done), seqs_acc=int(rows_acc))


def run_reference(args):
    from speculative_decoding_verification_gqa_gb300 import synth
    _, rank, _ = rank_info()
    if rank != 0:  # the reference arm runs on rank 0 only; the other ranks exit at once
        return
    w, T, D, p = workload(args)
    x = synth.attn_inputs(w, args.seed, seq_lens=T, draft_len=D)
    a = synth.accept_inputs(w, args.seed, draft_len=D, p=p)
    per_step = min(10.0, max(0.05, 150.0 / max(1, args.steps + args.warmup)))
    for s in range(args.warmup):
        cpu_oracle_sample(w, x, a, per_step, args.seed + 10007 + s, acc_rows=8)
    t_steps = []
    secs = 0.0
    rows = 0
    threads = 1
    acc = []
    for s in range(args.steps):
        r = cpu_oracle_sample(w, x, a, per_step, args.seed + s, acc_rows=8)
        t_steps.append(r["t_step"])
        secs += r["seconds"]
        rows += r["rows"]
        threads = r["threads"]
        acc.append(r["acc_per_s"] * r["t_step"])
    kv_bytes, _ = algorithmic_bytes(w, T, D)
    t_mean = float(np.mean(t_steps))
    gbs = kv_bytes / t_mean / 1e9
    sample = ("each step: a random sample of the workload's (window row, head) outputs "
              "through the fp64 oracle (~%.2f s) plus acceptance of sampled sequences, "
              "extrapolated to the whole step by the fraction of keys / logit rows done; "
              "%d outputs over %d steps, %.1f s of oracle time"
              % (per_step, rows, args.steps, secs))
    line = {"impl": "reference", "metric": METRIC, "value": round(gbs, 5), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * t_mean, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": describe(w, T, D), "parallelism": "host cores, OpenMP"},
            "accepted_tokens_per_s": round(float(np.mean(acc)) / t_mean, 4),
            "cpu_baseline": {"value": round(gbs, 5), "unit": "GB/s", "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(gbs, 5), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# DRAM bytes (read + written) per launch of the attention kernel, from one ncu capture per
# workload (dram__bytes_read.sum + dram__bytes_write.sum), keyed by (config, D override,
# kernel) with the kernel_source_hash() of the sources captured: an entry whose hash is not
# the current one reads as None.
NCU_TRAFFIC = {
    ("c2", None, "tcgen05"): ("7be090ecd712d963", 549_204_480 + 2_689_280),
    ("c3", None, "tcgen05"): ("7be090ecd712d963", 542_727_168 + 5_724_672),
    ("c4", 15, "tcgen05"): ("7be090ecd712d963", 1_086_250_496 + 2_968_832),
    ("c4", 16, "tcgen05"): ("7be090ecd712d963", 1_089_450_496 + 9_586_688),
    ("c4", 31, "tcgen05"): ("7be090ecd712d963", 1_263_172_096 + 15_799_296),
    ("c5", None, "tcgen05"): ("7be090ecd712d963", 9_004_360_448 + 6_521_600),
}


class Rig:
    """One workload's inputs on the device (and in pinned host memory for the end-to-end
    figures), its outputs and workspaces, and the step: spec_verify_attn + spec_accept."""


def build_rig(sv, synth, w, T, D, p, seed, dev, pinned=True):
    import torch
    r = Rig()
    r.x = x = synth.attn_inputs(w, seed, seq_lens=T, draft_len=D)
    r.a = a = synth.accept_inputs(w, seed, draft_len=D, p=p)

    def host_tensor(arr, dtype):
        t = torch.from_numpy(arr.view(np.int16) if dtype == torch.bfloat16 else arr)
        if dtype == torch.bfloat16:
            t = t.view(torch.bfloat16)
        return t.pin_memory() if pinned else t

    r.kvdt = kvdt = torch.uint8 if w.kv_dtype == "fp8_e4m3" else torch.bfloat16
    lgdt = torch.bfloat16 if w.logits_dtype == "bf16" else torch.float32
    h = {"q": host_tensor(x["q"], torch.bfloat16), "k": host_tensor(x["k"], kvdt),
         "v": host_tensor(x["v"], kvdt), "T": host_tensor(x["seq_lens"], torch.int32),
         "D": host_tensor(x["draft_len"], torch.int32),
         "logits": host_tensor(a["logits"], lgdt),
         "draft": host_tensor(a["draft_tokens"], torch.int32)}
    if x["kv_scale"] is not None:
        h["sc"] = host_tensor(x["kv_scale"], torch.float32)
    r.h = h
    r.d = d = {k: t.to(dev) for k, t in h.items()}
    r.out = torch.empty_like(d["q"])
    r.al = torch.empty(w.B, dtype=torch.int32, device=dev)
    r.nt = torch.empty(w.B, dtype=torch.int32, device=dev)
    r.md, r.ms = int(D.max()), int(T.max())
    r.desc = sv.api.attn_desc(d["q"], d["k"], w.B, r.md, r.ms)
    r.ws_attn = sv.new_workspace(sv.verify_workspace_bytes(r.desc), dev)
    r.ws_acc = sv.new_workspace(sv.accept_workspace_bytes(w.B, r.md, w.V), dev)
    stream = torch.cuda.current_stream()

    def step():
        sv.spec_verify_attn(d["q"], d["k"], d["v"], d["T"], d["D"], max_draft_len=r.md,
                            max_seq_len=r.ms, kv_scale=d.get("sc"), out=r.out,
                            workspace=r.ws_attn, stream=stream)
        sv.spec_accept(d["logits"], d["draft"], d["D"], max_draft_len=r.md, accept_len=r.al,
                       next_token=r.nt, workspace=r.ws_acc, stream=stream)

    r.step = step
    return r


def warm_up(step, n_min, seconds=0.3):
    """At least n_min steps and `seconds` of them. Returns the number run."""
    import torch
    n = 0
    t0 = time.perf_counter()
    while n < n_min or time.perf_counter() - t0 < seconds:
        step()
        n += 1
        if n % 16 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    return n


def timed_steps(step, stream, K):
    """ms per step over exactly K steps: CUDA events on the launching stream around the
    loop, synchronised on both sides."""
    import torch
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(K):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / K


def timed_attention(sv, step, stream, K):
    """Mean duration (ms) of the attention kernel over K more steps, from events the library
    records just before and after it on the call's stream."""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    for a_, b_ in ev:  # create the events the library records into
        a_.record(stream)
        b_.record(stream)
    torch.cuda.synchronize()
    for a_, b_ in ev:
        sv.set_profile_events(a_, b_)
        step()
    torch.cuda.synchronize()
    sv.set_profile_events(None, None)
    return float(np.mean([a_.elapsed_time(b_) for a_, b_ in ev]))


def measure_config(sv, synth, cfg, Dv, seed, dev, K, W, attn_kernel, src_hash,
                   row_pairs=False):
    """The step of another workload: attention and step time, K/V GB/s, verified query
    tokens/s, accepted tokens/s and the attention kernel's roofline."""
    import torch
    w = synth.CONFIGS[cfg]
    T, D, p = synth.lengths(w, seed, D=Dv)
    rig = build_rig(sv, synth, w, T, D, p, seed, dev, pinned=False)
    stream = torch.cuda.current_stream()
    warm_up(rig.step, W)
    if sv.workspace_status(rig.ws_attn) != 0 or sv.workspace_status(rig.ws_acc) != 0:
        raise RuntimeError("device-side check failed on %s" % cfg)
    accepted = int(rig.al.sum().item())
    ms_step = timed_steps(rig.step, stream, K)
    attn_ms = timed_attention(sv, rig.step, stream, K)
    kv, qo = algorithmic_bytes(w, T, D)
    fl = flops(w, T, D)
    hbm, tf, _ = peaks()
    W_rows = int(np.sum(D.astype(np.int64) + 1))
    rec = {"workload": describe(w, T, D), "steps": K, "attn_us": round(attn_ms * 1e3, 2),
           "step_us": round(ms_step * 1e3, 2),
           "attn_kv_GB_per_s": round(kv / (attn_ms / 1e3) / 1e9, 1),
           "step_kv_GB_per_s": round(kv / (ms_step / 1e3) / 1e9, 1),
           "verified_query_tokens_per_s": round(W_rows / (ms_step / 1e3), 1),
           "accepted_tokens_per_s": round(accepted / (ms_step / 1e3), 1),
           "mean_accept_len": round(accepted / w.B, 3),
           "attn_tflops": round(fl / (attn_ms / 1e3) / 1e12, 1),
           "roofline": roofline_record(kv, qo, fl, attn_ms / 1e3, hbm, tf, w.kv_dtype,
                                       attn_kernel,
                                       None if row_pairs else
                                       ncu_traffic(cfg, Dv, attn_kernel, src_hash))}
    if row_pairs:
        rec["kernel"] = "row pairs (one CTA per sequence and KV head, both 128-row tiles)"
    del rig
    torch.cuda.empty_cache()
    return rec


def run_ours(args):
    import torch
    import torch.distributed as dist

    import speculative_decoding_verification_gqa_gb300 as sv
    from speculative_decoding_verification_gqa_gb300 import build, synth

    world, rank, local = rank_info()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    if rank == 0:
        build.build()
    if world > 1:
        dist.barrier()
    sv.load_library()
    if args.kernel != "auto":
        sv.set_attn_kernel(1 if args.kernel == "mma" else 2)
    sv.api.set_row_pairs(args.row_pairs)
    sv.api.set_kv_rings(args.kv_rings)
    attn_kernel = {1: "mma.sync", 2: "tcgen05"}[_active_kernel(sv)]

    w, T, D, p = workload(args)
    seed = replica_seed(args.seed, rank)  # each rank verifies its own batch (replicas)
    rig = build_rig(sv, synth, w, T, D, p, seed, dev, pinned=True)
    x, a, h, d = rig.x, rig.a, rig.h, rig.d
    out, al, nt, ws_attn, ws_acc = rig.out, rig.al, rig.nt, rig.ws_attn, rig.ws_acc
    md, ms, desc, step = rig.md, rig.ms, rig.desc, rig.step
    kvdt = rig.kvdt
    kv_bytes, qo_bytes = algorithmic_bytes(w, T, D)
    fl = flops(w, T, D)
    stream = torch.cuda.current_stream()
    if args.only_step:  # W + K plain steps, nothing else (what a profiler captures)
        for _ in range(args.warmup + args.steps):
            step()
        torch.cuda.synchronize()
        st = (sv.workspace_status(ws_attn), sv.workspace_status(ws_acc))
        if rank == 0:
            print(json.dumps({"only_step": True, "workload": describe(w, T, D),
                              "steps": args.warmup + args.steps, "status": st}), flush=True)
        if st != (0, 0):
            raise RuntimeError("device-side check failed")
        return

    # warm-up: at least W steps and 0.3 s, so the clocks are up before the timed region
    clocks = ClockSampler(dev.index)
    if rank == 0:
        clocks.start()
    n_warm = warm_up(step, max(3, args.warmup))
    if sv.workspace_status(ws_attn) != 0 or sv.workspace_status(ws_acc) != 0:
        raise RuntimeError("device-side check failed during warm-up")
    accepted_per_step = int(al.sum().item())

    # Two timed regions. (1) The step itself: CUDA events only around the whole loop, so
    # nothing breaks the programmatic overlap between the step's kernels. (2) The same K
    # steps again with events recorded inside the library just before and after the
    # attention kernel, for its duration (the roofline); those events cost the step its
    # launch overlap, so region 2 is not the step time.
    K = args.steps
    if world > 1:
        dist.barrier()
    ms_step = timed_steps(step, stream, K)
    attn_ms = timed_attention(sv, step, stream, K)
    if world > 1:
        dist.barrier()
    clk = clocks.stop() if rank == 0 else None

    # The same step through spec_verify_attn_host_lengths (lengths also in host memory, as
    # an engine's scheduler holds them: the work plan travels with the attention launch and
    # no planning kernel runs). Timed like the step, without events inside it.
    T_host = torch.from_numpy(x["seq_lens"].astype(np.int32))
    D_host = torch.from_numpy(x["draft_len"].astype(np.int32))

    def step_host_lengths():
        sv.spec_verify_attn_host_lengths(d["q"], d["k"], d["v"], d["T"], d["D"], T_host, D_host,
                                         max_draft_len=md, max_seq_len=ms,
                                         kv_scale=d.get("sc"), out=out, workspace=ws_attn,
                                         stream=stream)
        sv.spec_accept(d["logits"], d["draft"], d["D"], max_draft_len=md, accept_len=al,
                       next_token=nt, workspace=ws_acc, stream=stream)

    for _ in range(3):
        step_host_lengths()
    torch.cuda.synchronize()
    h0 = torch.cuda.Event(enable_timing=True)
    h1 = torch.cuda.Event(enable_timing=True)
    h0.record(stream)
    for _ in range(K):
        step_host_lengths()
    h1.record(stream)
    torch.cuda.synchronize()
    if sv.workspace_status(ws_attn) != 0:
        raise RuntimeError("device-side check failed in the host-lengths step")
    ms_step_hl = h0.elapsed_time(h1) / K

    # split of a step between the two calls (separate pass, after the timed region)
    K3 = max(1, min(K, 200))
    e3 = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K3)]
    for i in range(K3):
        e3[i][0].record(stream)
        sv.spec_verify_attn(d["q"], d["k"], d["v"], d["T"], d["D"], max_draft_len=md,
                            max_seq_len=ms, kv_scale=d.get("sc"), out=out, workspace=ws_attn,
                            stream=stream)
        e3[i][1].record(stream)
        sv.spec_accept(d["logits"], d["draft"], d["D"], max_draft_len=md, accept_len=al,
                       next_token=nt, workspace=ws_acc, stream=stream)
        e3[i][2].record(stream)
    torch.cuda.synchronize()
    verify_ms = float(np.median([e[0].elapsed_time(e[1]) for e in e3]))
    accept_ms = float(np.median([e[1].elapsed_time(e[2]) for e in e3]))

    # Acceptance's share of the step: the step loop against the same loop with the verify
    # call alone, both without events inside (the events around each call above expose
    # every launch; in the step the launches overlap their predecessors)
    def verify_only():
        sv.spec_verify_attn(d["q"], d["k"], d["v"], d["T"], d["D"], max_draft_len=md,
                            max_seq_len=ms, kv_scale=d.get("sc"), out=out, workspace=ws_attn,
                            stream=stream)

    for _ in range(3):
        verify_only()
    accept_in_step_ms = ms_step - timed_steps(verify_only, stream, K)

    # draft signals (confidence, entropy per row) over the step's logits matrix, as a
    # stand-in for the draft model's logits of the same shape (not part of the step)
    rows_l, V_l = d["logits"].shape
    sig_c = torch.empty(rows_l, dtype=torch.float32, device=dev)
    sig_e = torch.empty(rows_l, dtype=torch.float32, device=dev)
    ws_sig = sv.new_workspace(sv.signals_workspace_bytes(rows_l, V_l), dev)
    for _ in range(3):
        sv.spec_draft_signals(d["logits"], confidence=sig_c, entropy=sig_e, workspace=ws_sig,
                              stream=stream)
    es = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K3)]
    for i in range(K3):
        es[i][0].record(stream)
        sv.spec_draft_signals(d["logits"], confidence=sig_c, entropy=sig_e, workspace=ws_sig,
                              stream=stream)
        es[i][1].record(stream)
    torch.cuda.synchronize()
    signals_ms = float(np.median([e[0].elapsed_time(e[1]) for e in es]))
    logits_bytes = d["logits"].numel() * d["logits"].element_size()

    # The two logits scans beside torch's own row reductions over the same logits, each
    # call after L2 is evicted (a buffer four times L2's size read), as a yardstick for a
    # one-shot read of this size (not part of the step)
    # four times L2: reading it also keeps the GPU busy for longer than the host needs to
    # enqueue the timed call, so the events time the call, not the host
    flush_l = torch.ones(int(4 * L2_BYTES) // 4, dtype=torch.float32, device=dev)
    sink_l = torch.empty((), dtype=torch.float32, device=dev)
    scans = {
        "spec_accept": lambda: sv.spec_accept(d["logits"], d["draft"], d["D"], max_draft_len=md,
                                              accept_len=al, next_token=nt, workspace=ws_acc,
                                              stream=stream),
        "spec_draft_signals": lambda: sv.spec_draft_signals(d["logits"], confidence=sig_c,
                                                            entropy=sig_e, workspace=ws_sig,
                                                            stream=stream),
        "torch_argmax_dim1": lambda: torch.argmax(d["logits"], dim=1),
        "torch_amax_dim1": lambda: torch.amax(d["logits"], dim=1),
    }
    logits_scan = {}
    for name, fn in scans.items():
        fn()
        ec = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K3)]
        for i in range(K3):
            sink_l.copy_(flush_l.sum())
            ec[i][0].record(stream)
            fn()
            ec[i][1].record(stream)
        torch.cuda.synchronize()
        logits_scan[name + "_us"] = round(
            1e3 * float(np.median([a_.elapsed_time(b_) for a_, b_ in ec])), 2)
    logits_scan["bytes"] = logits_bytes
    logits_scan["note"] = ("each call after L2 is evicted (a read of 4x L2's size); torch's "
                           "reductions read the same logits; not part of the step")

    # distribution-preserving acceptance on the step's shapes: the step's target logits
    # plus drafter logits at every draft position (not part of the step)
    side_stoch = None
    if args.side_stochastic:
        xs = synth.stochastic_inputs(w, seed + 7, draft_len=D)
        dts = torch.bfloat16 if xs["target_logits"].dtype == np.uint16 else torch.float32
        as_dev = lambda arr: (torch.from_numpy(arr.view(np.int16)).view(torch.bfloat16)
                              if arr.dtype == np.uint16 else torch.from_numpy(arr)).to(dev)
        st_in = [as_dev(xs["target_logits"]), as_dev(xs["draft_logits"]),
                 torch.from_numpy(xs["draft_tokens"]).to(dev),
                 torch.from_numpy(xs["draft_len"]).to(dev),
                 torch.from_numpy(xs["u_accept"]).to(dev), torch.from_numpy(xs["u_sample"]).to(dev)]
        st_out = (torch.empty(w.B, dtype=torch.int32, device=dev),
                  torch.empty(w.B, dtype=torch.int32, device=dev))
        ws_st = sv.new_workspace(256, dev)
        st_call = lambda: sv.spec_accept_stochastic(*st_in, max_draft_len=md, temperature=1.0,
                                                    accept_len=st_out[0], next_token=st_out[1],
                                                    workspace=ws_st, stream=stream)
        st_call()
        n_st = max(3, min(K3, 20))
        est = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n_st)]
        for i in range(n_st):
            sink_l.copy_(flush_l.sum())
            est[i][0].record(stream)
            st_call()
            est[i][1].record(stream)
        torch.cuda.synchronize()
        if sv.workspace_status(ws_st) != 0:
            raise RuntimeError("device-side check failed in the stochastic acceptance")
        st_ms = float(np.median([a_.elapsed_time(b_) for a_, b_ in est]))
        st_bytes = sum(t.numel() * t.element_size() for t in st_in[:2])
        # rows read: per sequence the (target, drafter) pairs examined (min(AL, D) of
        # them) and, when every draft was kept, the target's last row
        alh = st_out[0].cpu().numpy().astype(np.int64)
        Dn = D.astype(np.int64)
        row_b = V_l * (2 if dts == torch.bfloat16 else 4)
        st_read = int(np.sum(2 * np.minimum(alh, Dn) + (alh == Dn + 1)) * row_b)
        side_stoch = {"ms": round(st_ms, 5), "logits_bytes_allocated": st_bytes,
                      "bytes_examined": st_read,
                      "GB_per_s_examined": round(st_read / (st_ms / 1e3) / 1e9, 1),
                      "mean_accept_len": round(float(st_out[0].float().mean()), 3),
                      "max_accept_len": int(alh.max()),
                      "dtype": str(dts).replace("torch.", ""),
                      "note": "spec_accept_stochastic (temperature 1) on the step's target "
                              "logits and drafter logits at every draft position, L2 "
                              "evicted before each call; one cluster of 8 CTAs per "
                              "sequence; rows after the first rejection are not read; "
                              "not part of the step"}
        del st_in, xs
    del flush_l

    # sliding-window verify attention on the same inputs (not part of the step)
    side_win = None
    if args.side_window > 0:
        Wn = args.side_window
        out_w = torch.empty_like(out)
        ws_w = sv.new_workspace(sv.verify_workspace_bytes(
            sv.api.attn_desc(d["q"], d["k"], w.B, md, ms, sliding_window=Wn)), dev)

        def win_call():
            sv.spec_verify_attn(d["q"], d["k"], d["v"], d["T"], d["D"], max_draft_len=md,
                                max_seq_len=ms, kv_scale=d.get("sc"), out=out_w, workspace=ws_w,
                                sliding_window=Wn, stream=stream)

        for _ in range(3):
            win_call()
        ew = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K3)]
        for e in ew:  # create the events the library records into
            e[2].record(stream)
            e[3].record(stream)
        # the window's K/V may fit in L2: evict them before each call by reading a buffer
        # twice L2's size (reads leave clean lines, so no write-back lands in the call)
        flush = torch.ones(int(2 * L2_BYTES) // 4, dtype=torch.float32, device=dev)
        sink = torch.empty((), dtype=torch.float32, device=dev)
        for i in range(K3):
            sink.copy_(flush.sum())
            ew[i][0].record(stream)
            sv.set_profile_events(ew[i][2], ew[i][3])
            win_call()
            ew[i][1].record(stream)
        sv.set_profile_events(None, None)
        torch.cuda.synchronize()
        if sv.workspace_status(ws_w) != 0:
            raise RuntimeError("device-side check failed in the sliding-window call")
        win_ms = float(np.median([e[0].elapsed_time(e[1]) for e in ew]))
        win_attn_ms = float(np.median([e[2].elapsed_time(e[3]) for e in ew]))
        kvw, qow = algorithmic_bytes(w, T, D, window=Wn)
        side_win = {"window": Wn, "verify_call_ms": round(win_ms, 5),
                    "attn_ms": round(win_attn_ms, 5), "kv_bytes": kvw,
                    "GB_per_s": round((kvw + qow) / (win_ms / 1e3) / 1e9, 1),
                    "attn_GB_per_s": round((kvw + qow) / (win_attn_ms / 1e3) / 1e9, 1),
                    "attn_frac": round((kvw + qow) / (win_attn_ms / 1e3) / 1e9 / peaks()[0], 4),
                    "note": "spec_verify_attn with sliding_window on the step's inputs, L2 "
                            "evicted before each call; verify_call_ms = plan + attention + "
                            "combine, attn_ms = the attention kernel alone; bytes = K/V "
                            "positions max(0, T-W+1)..T+D plus Q and out; not part of the "
                            "step"}
        del flush

    # verify attention over a paged copy of the same cache (not part of the step)
    side_paged = None
    if args.side_block > 0:
        pg = synth.paged_layout(x, args.side_block, seed + 5, spare_blocks=256)
        to_dev = (lambda a: torch.from_numpy(a).to(dev)) if kvdt == torch.uint8 else \
            (lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev))
        kp, vp = to_dev(pg["k_pages"]), to_dev(pg["v_pages"])
        bt = torch.from_numpy(pg["block_table"]).to(dev)
        del pg
        out_p = torch.empty_like(out)
        ws_p = sv.new_workspace(sv.verify_workspace_bytes(desc), dev)

        def paged_call():
            sv.spec_verify_attn_paged(d["q"], kp, vp, bt, d["T"], d["D"], max_draft_len=md,
                                      max_seq_len=ms, kv_scale=d.get("sc"), out=out_p,
                                      workspace=ws_p, stream=stream)

        for _ in range(3):
            paged_call()
        ep = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K3)]
        for e in ep:
            e[2].record(stream)
            e[3].record(stream)
        for i in range(K3):
            ep[i][0].record(stream)
            sv.set_profile_events(ep[i][2], ep[i][3])
            paged_call()
            ep[i][1].record(stream)
        sv.set_profile_events(None, None)
        torch.cuda.synchronize()
        if sv.workspace_status(ws_p) != 0:
            raise RuntimeError("device-side check failed in the paged call")
        p_ms = float(np.median([e[0].elapsed_time(e[1]) for e in ep]))
        p_attn = float(np.median([e[2].elapsed_time(e[3]) for e in ep]))
        side_paged = {"block_size": args.side_block, "verify_call_ms": round(p_ms, 5),
                      "attn_ms": round(p_attn, 5),
                      "attn_GB_per_s": round((kv_bytes + qo_bytes) / (p_attn / 1e3) / 1e9, 1),
                      "attn_frac": round((kv_bytes + qo_bytes) / (p_attn / 1e3) / 1e9
                                         / peaks()[0], 4),
                      "note": "spec_verify_attn_paged on the step's K/V cut into blocks at "
                              "seeded random slots of a pool with 256 spare blocks; inputs "
                              "larger than L2; not part of the step"}
        del kp, vp

    # end to end: pinned host inputs -> device, step, result back to pinned host memory
    e2e = None
    if not args.no_e2e:
        res_h = {"al": torch.empty(w.B, dtype=torch.int32).pin_memory(),
                 "nt": torch.empty(w.B, dtype=torch.int32).pin_memory(),
                 "out": torch.empty(out.shape, dtype=out.dtype).pin_memory()}
        h2d = sum(t.numel() * t.element_size() for t in h.values())
        d2h = sum(t.numel() * t.element_size() for t in res_h.values())
        K2 = max(1, min(K, 200))

        def e2e_step():
            for k_, t in h.items():
                d[k_].copy_(t, non_blocking=True)
            step()
            res_h["al"].copy_(al, non_blocking=True)
            res_h["nt"].copy_(nt, non_blocking=True)
            res_h["out"].copy_(out, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(K2):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1) / K2
        e2e = {"ms": e2e_ms, "h2d": h2d, "d2h": d2h, "steps": K2}

        # The same with the cached prefix resident on the device, as across decoding steps:
        # each step uploads only what is new (the window's Q rows, the window's K/V rows,
        # lengths, drafts, logits; the window rows travel in one pinned buffer and are
        # scattered into the cache on the device) and reads back the same results.
        qo_h, ko_h = synth.packed_offsets(x["seq_lens"], x["draft_len"])
        win_rows = np.concatenate([np.arange(ko_h[b] + T[b], ko_h[b + 1])
                                   for b in range(len(T))]).astype(np.int64)
        win_idx = torch.from_numpy(win_rows).to(dev)
        hk = h["k"].view(h["k"].shape[0], -1)
        hv = h["v"].view(h["v"].shape[0], -1)
        win_h = torch.cat([hk[win_rows], hv[win_rows]]).pin_memory()
        win_d = torch.empty(win_h.shape, dtype=win_h.dtype, device=dev)
        small = ("q", "T", "D", "logits", "draft") + (("sc",) if "sc" in h else ())
        h2d_r = win_h.numel() * win_h.element_size() + sum(
            h[k_].numel() * h[k_].element_size() for k_ in small)
        nw = len(win_rows)

        def e2e_resident_step():
            for k_ in small:
                d[k_].copy_(h[k_], non_blocking=True)
            win_d.copy_(win_h, non_blocking=True)
            d["k"].view(d["k"].shape[0], -1).index_copy_(0, win_idx, win_d[:nw])
            d["v"].view(d["v"].shape[0], -1).index_copy_(0, win_idx, win_d[nw:])
            step()
            res_h["al"].copy_(al, non_blocking=True)
            res_h["nt"].copy_(nt, non_blocking=True)
            res_h["out"].copy_(out, non_blocking=True)

        for _ in range(2):
            e2e_resident_step()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        e0.record(stream)
        for _ in range(K2):
            e2e_resident_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e["ms_resident"] = e0.elapsed_time(e1) / K2
        e2e["h2d_resident"] = h2d_r

    # the other workloads, each through the same step (not part of the headline)
    per_config = None
    src_hash = kernel_source_hash()
    if args.per_config != "none" and args.config == "c2" and args.D is None:
        per_config = {}
        for item in args.per_config.split(","):
            parts = item.split(":")
            cfg = parts[0]
            Dv = int(parts[1]) if len(parts) > 1 and parts[1] else None
            pairs = len(parts) > 2 and parts[2] == "pairs"
            key = cfg + ("_D%d" % Dv if Dv is not None else "") + ("_row_pairs" if pairs else "")
            prev_pairs = sv.api.set_row_pairs(1 if pairs else args.row_pairs)
            per_config[key] = measure_config(sv, synth, cfg, Dv, seed, dev,
                                             args.per_config_steps, max(3, args.warmup),
                                             attn_kernel, src_hash, row_pairs=pairs)
            sv.api.set_row_pairs(prev_pairs)

    # max over ranks
    ms_step, attn_ms, e2e_ms, e2e_res_ms, ms_step_hl = max_over_ranks(
        [ms_step, attn_ms, e2e["ms"] if e2e else 0.0, e2e["ms_resident"] if e2e else 0.0,
         ms_step_hl], device=dev)

    if rank == 0:
        hbm, tf, src = peaks()
        sec = ms_step / 1e3
        value = whole_job_rate(world, kv_bytes, sec) / 1e9
        cpu = None
        if not args.no_cpu_baseline:
            r = cpu_oracle_sample(w, x, a, args.cpu_seconds, args.seed)
            cpu = {"value": round(r["gbs"], 5), "unit": "GB/s", "cores": r["threads"],
                   "kind": "oracle",
                   "sample": "fp64 oracle on %d random (window row, head) outputs (%.2f%% of "
                             "the attention's key visits) and the acceptance of %d logit rows "
                             "(%.1f%%), %.1f s, extrapolated to one whole step (%.1f s)"
                             % (r["rows"], 100 * r["f_attn"], r["seqs_acc"], 100 * r["f_acc"],
                                r["seconds"], r["t_step"])}
        W = D.astype(np.int64) + 1
        try:  # the attention call's work plan, as the library makes it for these lengths
            pl = sv.plan_preview(sv.api.attn_desc(d["q"], d["k"], w.B, md, ms), T, D,
                                 num_sms=torch.cuda.get_device_properties(dev).multi_processor_count,
                                 attn_kernel=2 if attn_kernel == "tcgen05" else 1)
            attn_plan = {"units": pl["num_units"], "tiles": pl["total_tiles"],
                         "ctas": pl["num_ctas"], "ctas_per_unit": pl["unit_ctas"] or None,
                         "policy": ("%d CTA(s) per unit" % pl["unit_ctas"]) if pl["unit_ctas"]
                                   else "one tile line split over the CTAs"}
        except sv.SpecVerifyError:
            attn_plan = None
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": K, "warmup": n_warm, "ms_per_step": round(ms_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": ("fp8_e4m3 (QK^T: e4m3 x e4m3, Q as two e4m3 terms; PV: f16), fp32 accum"
                      if attn_kernel == "tcgen05" else "fp8_e4m3->f16 mma, fp32 accum")
                     if w.kv_dtype == "fp8_e4m3"
                     else "bf16 mma, fp32 accum",
            "data": "synthetic",
            "config": {"workload": describe(w, T, D),
                       "l2": "inputs larger than L2 (%.0f MB K/V + %.0f MB logits vs 129 MB L2)"
                             % (kv_bytes / 1e6, logits_bytes / 1e6)
                             if kv_bytes > L2_BYTES else "inputs smaller than L2",
                       "parallelism": "replicas" if world > 1 else "1 GPU"},
            "accepted_tokens_per_s": round(whole_job_rate(world, accepted_per_step, sec), 1),
            "verified_query_tokens_per_s": round(whole_job_rate(world, int(W.sum()), sec), 1),
            "kv_bytes_per_step": kv_bytes,
            "attn_kernel": attn_kernel,
            "attn_plan": attn_plan,
            "attn_ms": round(attn_ms, 5),
            "verify_call_ms": round(verify_ms, 5),
            "accept_call_ms": round(accept_ms, 5),
            "accept_in_step_ms": round(accept_in_step_ms, 5),
            "draft_signals": {"ms": round(signals_ms, 5),
                              "GB_per_s": round(logits_bytes / (signals_ms / 1e3) / 1e9, 1),
                              "rows": rows_l, "vocab": V_l,
                              "note": "spec_draft_signals on a logits matrix of the step's "
                                      "shape; not part of the step"},
            "logits_scans": logits_scan,
            "stochastic_accept": side_stoch,
            "host_lengths": {
                "ms_per_step": round(ms_step_hl, 5),
                "value": round(whole_job_rate(world, kv_bytes, ms_step_hl / 1e3) / 1e9, 2),
                "unit": "GB/s",
                "note": "the same step through spec_verify_attn_host_lengths (lengths also "
                        "in host memory: the work plan is made on the host and passed "
                        "with the attention launch, no planning kernel)"},
            "sliding_window": side_win,
            "paged": side_paged,
            "attn_tflops": round(fl / (attn_ms / 1e3) / 1e12, 2),
            "roofline": dict(roofline_record(kv_bytes, qo_bytes, fl, attn_ms / 1e3, hbm, tf,
                                             w.kv_dtype, attn_kernel,
                                             ncu_traffic(args.config, args.D, attn_kernel,
                                                         src_hash)),
                             traffic_unit="bytes per launch (ncu), null unless captured "
                                          "from the current kernel sources",
                             kernel_source_hash=src_hash,
                             peak_source=src + " (HBM: STREAM-style copy; tensor: cuBLAS "
                                               "bf16 burst, e4m3 = bf16 x 2 nominal)",
                             kernel="verify attention (%s)" % attn_kernel,
                             timing="CUDA events recorded just before and after the "
                                    "attention kernel on its stream, averaged over a "
                                    "second pass of the K steps (the step time comes "
                                    "from a pass without them)"),
            "per_config": per_config,
            "cpu_baseline": cpu,
            "e2e": None if e2e is None else {
                "value": round(whole_job_rate(world, kv_bytes, e2e_ms / 1e3) / 1e9, 2),
                "unit": "GB/s",
                "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                "ms_per_step": round(e2e_ms, 4), "steps": e2e["steps"],
                "note": "every step uploads all of its inputs, the whole K/V cache included"},
            "e2e_resident_cache": None if e2e is None else {
                "value": round(whole_job_rate(world, kv_bytes, e2e_res_ms / 1e3) / 1e9, 2),
                "unit": "GB/s",
                "h2d_bytes_per_step": e2e["h2d_resident"], "d2h_bytes_per_step": e2e["d2h"],
                "ms_per_step": round(e2e_res_ms, 4), "steps": e2e["steps"],
                "note": "the cached prefix stays on the device across steps; every step "
                        "uploads its new inputs (window Q and K/V rows, lengths, drafts, "
                        "logits) and reads back the acceptance results and the attention "
                        "output"},
            "clocks": clk,
            # plan, attention, combine (verify call); argmax + acceptance (accept call)
            "gpu_launches": 4 * K,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def _active_kernel(sv):
    lib = sv.load_library()
    cur = lib.sv_set_attn_kernel(0)
    lib.sv_set_attn_kernel(cur)
    if cur in (1, 2):
        return cur
    prev = lib.sv_set_attn_kernel(2)
    if prev < 0:
        return 1
    lib.sv_set_attn_kernel(prev)
    return 2


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
