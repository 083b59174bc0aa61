"""The benchmark's multi-rank harness on CPU (gloo, world size 2): each rank
runs its own replica with its own seed -- here the CPU oracle over the rank's
own small workload, every invariant checked after every step -- elapsed time
is the max over ranks and work is summed.  No GPU and no data-path collective
are involved."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    import bench
    import skv_workload as wl
    ws, r, local = bench.dist_env()
    dist = bench.init_dist(ws)
    w = bench.rank_seed(wl.WORKLOADS["c1_tiny"], r)
    # a replica's input: this rank's first Top-k step
    topk = wl.TopkStream(w, nthreads=1).step(0, [w.ctx] * w.B)
    # the rank's replica, driven on the CPU: the oracle over its own seeded
    # workload, checked against every invariant after every step
    import oracle_pins as op
    small = bench.rank_seed(wl.Workload("replica", B=2, L=2, ctx=600, k=64, S=100, steps=4, fresh=0.3), r)
    rows = op.check_invariants(small)
    elapsed, moved, tokens = bench.reduce_results(dist, 1.0 + r, float(rows), 10.0)
    out.put((r, (ws, r, local), w.seed, int(topk.sum()), elapsed, moved, tokens, rows))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_harness_reduces_and_seeds_independently():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, env0, seed0, sum0, e0, m0, t0, g0), (r1, env1, seed1, sum1, e1, m1, t1, g1) = res
    assert env0 == (2, 0, 0) and env1 == (2, 1, 1)
    assert seed0 != seed1 and sum0 != sum1          # independent replicas
    assert g0 > 0 and g1 > 0                         # each replica moved rows of its own
    assert e0 == e1 == 2.0                           # max over ranks
    assert m0 == m1 == float(g0 + g1) and t0 == t1 == 20.0    # work summed over ranks


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.init_dist(1) is None
    assert bench.reduce_results(None, 1.5, 2.0, 3.0) == (1.5, 2.0, 3.0)


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` (the CPU oracle, the one arm that runs without a GPU)
    prints one JSON line with the contract's keys."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--workload", "c1_tiny",
                        "--steps", "2", "--warmup", "3"], capture_output=True, text=True, timeout=300, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["config"]["workload"] == "c1_tiny"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
