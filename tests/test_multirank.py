"""The multi-rank path of bench.py on CPU: two gloo ranks on 127.0.0.1.

bench.py under torchrun runs one independent replica of the workload per GPU
(weak scaling, no collective on the data path).  The only cross-rank steps
are the barriers around the timed region and the max over ranks of the timed
durations; the reported throughput is every rank's work over the slowest
rank's time.  These tests run exactly those functions across two processes,
and the reference arm under torchrun (rank 0 alone prints, the other rank
exits 0 without work)."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


WORKER = r"""
import os, sys, json
sys.path.insert(0, %r)
import torch.distributed as dist
import bench
dist.init_process_group("gloo", init_method="env://")
rank, world, local = bench.dist_env()
ms = [4.0, 7.5][rank]                         # the two replicas' timed durations
bench.barrier(world)
worst = bench.max_over_ranks(ms, world)       # CPU tensor all-reduce (device=None)
rate = bench.whole_job_rate(3.0e12, worst, world, 1e12)
print(json.dumps({"rank": rank, "world": world, "max_ms": worst, "rate": rate}), flush=True)
bench.barrier(world)
dist.destroy_process_group()
""" % ROOT


def run_two_ranks(code):
    port = free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, "-c", code], env=env, cwd=ROOT,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err[-2000:]
        outs.append(out)
    return outs


def test_max_over_ranks_and_whole_job_rate():
    outs = run_two_ranks(WORKER)
    lines = [json.loads(o.strip().splitlines()[-1]) for o in outs]
    assert sorted(l["rank"] for l in lines) == [0, 1]
    for l in lines:
        assert l["world"] == 2
        assert l["max_ms"] == 7.5                          # both ranks see the slowest rank
        assert l["rate"] == pytest.approx(2 * 3.0 / 7.5e-3)  # 2 x 3 TFLOP over 7.5 ms


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
    bench.barrier(1)
    assert bench.whole_job_rate(1e9, 1.0, 1, 1e9) == pytest.approx(1000.0)


def test_reference_arm_under_torchrun_prints_once():
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "1", "--warmup", "3", "--prefill", "single_head"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0


CP_WORKER = r"""
import os, sys, json, math
sys.path.insert(0, %r)
import numpy as np
import torch
import torch.distributed as dist
import bench, oracle
from exact_attention_62_gb300.inputs import make_qkv
dist.init_process_group("gloo", init_method="env://")
rank, world, local = bench.dist_env()
out = {}
for name, (B, Hq, Hkv, Nq, Nk, d, causal) in {"prefill_causal": (1, 4, 2, 300, 300, 16, True),
                                              "prefill": (2, 2, 1, 130, 257, 8, False),
                                              "decode": (2, 4, 2, 1, 1000, 16, False)}.items():
    q, k, v = make_qkv(B, Hq, Hkv, Nq, Nk, d, seed=3)
    scale = 1.0 / math.sqrt(d)
    # this rank's key shard, and the partial result of every query row over it
    j0, j1 = rank * Nk // world, (rank + 1) * Nk // world
    rows = B * Hq * Nq
    o_p = torch.zeros(rows, d, dtype=torch.float64)
    l_p = torch.full((rows,), float("-inf"), dtype=torch.float64)
    r = 0
    for b in range(B):
        for hq in range(Hq):
            for i in range(Nq):
                m, l, acc = oracle.segment_state(q, k, v, causal, scale, b, hq, i, j0, j1)
                if l > 0:
                    o_p[r] = torch.from_numpy(acc / l)
                    l_p[r] = m + math.log(l)
                r += 1
    # the one exchange step, then the lse merge of the gathered partials
    o_all = [torch.empty_like(o_p) for _ in range(world)]
    l_all = [torch.empty_like(l_p) for _ in range(world)]
    dist.all_gather(o_all, o_p)
    dist.all_gather(l_all, l_p)
    o_m, l_m = oracle.merge_lse(torch.stack(o_all).numpy(), torch.stack(l_all).numpy())
    o_ref, l_ref = oracle.attn_fwd(q, k, v, causal, scale)
    o_ref = np.transpose(o_ref, (0, 2, 1, 3)).reshape(rows, d)      # [B, Hq, Nq, d] row order
    l_ref = np.asarray(l_ref).reshape(rows)
    fin = np.isfinite(l_ref)
    out[name] = {"dO": float(np.abs(o_m - o_ref).max()),
                 "dL": float(np.abs(l_m[fin] - l_ref[fin]).max()) if fin.any() else 0.0,
                 "inf_match": bool(np.array_equal(np.isfinite(l_m), fin))}
print(json.dumps({"rank": rank, "res": out}), flush=True)
dist.destroy_process_group()
""" % ROOT


def test_context_parallel_merge_over_gloo_ranks():
    """A context-parallel split (each rank holds half of the keys) needs one
    exchange: every rank's partial (o, lse) of every query row, all-gathered,
    then the lse merge of Lecture 11 section 6.2 step 3.  Two gloo ranks
    compute their shards' partials with the oracle (global causal rule, so
    some rows see no key of a shard: o = 0, lse = -inf), all-gather them and
    merge; the result equals the unsharded oracle to 1e-12 on each rank."""
    outs = run_two_ranks(CP_WORKER)
    for o in outs:
        res = json.loads(o.strip().splitlines()[-1])["res"]
        for name, r in res.items():
            assert r["inf_match"], name
            assert r["dO"] <= 1e-12 and r["dL"] <= 1e-12, (name, r)
