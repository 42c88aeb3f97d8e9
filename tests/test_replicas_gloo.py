"""Multi-GPU host logic on CPU: the prolog shards by tokens into independent replicas.  Two gloo
ranks check the benchmark's rendezvous, barrier and max-over-ranks timing, and that the
replicas' per-rank token shards reassemble the single-process result (oracle on CPU)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, local, w = bench._dist_setup(world)
    assert (r, local, w) == (rank, rank, world)
    bench._barrier(w)
    t_max = bench._max_over_ranks(1.0 + rank, w)          # max over ranks
    # each replica processes its own token shard of a tiny workload
    import oracle
    import synthetic
    from tests.gpu_util import oracle_inputs
    case = synthetic.small_mla_case("rep", B=4, S=1, He=64, Hcq=32, Hckv=32, N=2, D=128, Dr=32,
                                    block_num=1)
    inp = oracle_inputs(synthetic.make_mla_inputs(case), case.eps)
    shard = np.arange(rank, 4, world)
    from oracle.mla_prolog import mla_prolog_tokens
    q = mla_prolog_tokens(inp, shard)["query"]
    gathered = [None] * w
    dist.all_gather_object(gathered, (shard.tolist(), q))
    dist.destroy_process_group()
    out.put((rank, t_max, gathered))


@pytest.mark.timeout(300)
def test_two_gloo_replicas():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=240) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t_max, gathered in res:
        assert t_max == 2.0
    # the shards reassemble the single-process oracle result
    import oracle
    import synthetic
    from tests.gpu_util import oracle_inputs
    case = synthetic.small_mla_case("rep", B=4, S=1, He=64, Hcq=32, Hckv=32, N=2, D=128, Dr=32,
                                    block_num=1)
    full = oracle.mla_prolog(**oracle_inputs(synthetic.make_mla_inputs(case), case.eps))["query"]
    merged = np.empty_like(full)
    for shard, qpart in res[0][2]:
        merged[shard] = qpart
    np.testing.assert_array_equal(merged, full)


@pytest.mark.timeout(300)
def test_bench_gpus_flag_spawns_replicas():
    # `bench.py --gpus 2` without a launcher starts the two replicas itself (spawned processes
    # meeting over gloo on 127.0.0.1); the reference arm runs on rank 0 and reports both ranks
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    res = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                          "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "tiny"],
                         capture_output=True, text=True, timeout=280, env=env, cwd=root)
    assert res.returncode == 0, res.stderr[-3000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, res.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["cpu_baseline"]["value"] == line["value"]


def test_bench_rejects_world_size_mismatch():
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0")
    res = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                          "--gpus", "2", "--steps", "1"], capture_output=True, text=True,
                         timeout=120, env=env, cwd=root)
    assert res.returncode != 0 and "WORLD_SIZE" in (res.stderr + res.stdout)
