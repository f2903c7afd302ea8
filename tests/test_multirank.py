"""The multi-GPU path of the benchmark is N independent replicas (no data-path
collective): each rank verifies its own batch and the ranks only agree on the slowest
timing. These tests run that host logic as world_size-2 gloo process groups on the CPU."""
import os
import socket
import subprocess
import sys

import numpy as np
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    from speculative_decoding_verification_gqa_gb300 import synth
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w_, r_, l_ = bench.rank_info()
        # each rank reports its own step time; every rank must see the slowest one
        got = bench.max_over_ranks([1.0 + rank, 5.0 - rank, 0.0])
        # replicas: each rank's inputs come from its own seed
        seed = bench.replica_seed(0, rank)
        x = synth.attn_inputs(synth.CONFIGS["c1"], seed)
        out.put((rank, (w_, r_, l_), got, seed, x["q"][:4].copy()))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_distinct_batches():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in procs:
        r, info, got, seed, q = out.get(timeout=120)
        res[r] = (info, got, seed, q)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(2):
        assert res[r][0] == (2, r, r)
        assert res[r][1] == [2.0, 5.0, 0.0]  # element-wise max over both ranks
    assert res[0][2] != res[1][2]
    assert not np.array_equal(res[0][3], res[1][3])


def test_single_process_max_is_identity_and_job_rate_is_weak_scaling():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.0, 1.5]) == [3.0, 1.5]
    assert bench.whole_job_rate(4, 10.0, 2.0) == 20.0  # 4 ranks x 10 units in 2 s
    assert bench.replica_seed(7, 0) == 7


def test_reference_arm_runs_on_rank_zero_only():
    """Under torchrun every rank runs bench.py; the reference arm works on rank 0 alone and
    the others exit 0 at once without printing."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "c1", "--steps", "1", "--warmup", "0"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_line_has_the_contract_keys():
    """`bench.py --impl reference` prints one JSON line with the benchmark contract's keys,
    its cpu_baseline describing the run and an e2e object without copies."""
    import json
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "c1", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e", "impl"):
        assert k in d, k
    assert d["impl"] == "reference" and d["steps"] == 1 and d["warmup"] == 0
    assert d["value"] > 0 and d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert "workload" in d["config"]
