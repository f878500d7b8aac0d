"""The multi-rank host logic of bench.py, on CPU with two gloo ranks.

The path shards by batch with no data exchange ("replicas only", weak scaling):
every rank runs its own synthetic batch (seed = rank) of the same shape, every
timing is the slowest rank's (max over ranks), and the reference arm prints its
line on rank 0 only while the other ranks return without work.
"""

import argparse
import contextlib
import io
import json
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from synth import make_config
        ws, r, local = bench.dist_info()
        slowest = bench.max_over_ranks(10.0 + 5.0 * rank, "cpu")
        case = make_config("tiny_decode", seed=rank)
        # The reference arm on the tiny workload, with the oracle timing replaced by a
        # fixed sample so that the test stays short.
        bench.WORKLOAD = "tiny_decode"
        bench.cpu_oracle_rate = lambda c, budget_s=10.0: (1.5, 2, 2, 0.01)
        buf = io.StringIO()
        with contextlib.redirect_stdout(buf):
            bench.run_reference(argparse.Namespace(steps=2, warmup=1, gpus=world))
        dist.barrier()
        out_q.put(dict(rank=rank, ws=ws, r=r, local=local, slowest=slowest,
                       q=case.q.float().numpy().tolist(), q_shape=tuple(case.q.shape),
                       cache_shape=tuple(case.key_cache.shape),
                       lens=case.seq_lens.tolist(), printed=buf.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        res = sorted((q.get(timeout=240) for _ in range(2)), key=lambda d: d["rank"])
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert [p.exitcode for p in procs] == [0, 0]

    # Rank discovery from the launcher's environment.
    assert [(d["ws"], d["r"], d["local"]) for d in res] == [(2, 0, 0), (2, 1, 1)]
    # Every rank sees the slowest rank's time.
    assert [d["slowest"] for d in res] == [15.0, 15.0]
    # Weak scaling: same shapes per rank, different synthetic data per rank.
    assert res[0]["q_shape"] == res[1]["q_shape"]
    assert res[0]["cache_shape"] == res[1]["cache_shape"]
    assert res[0]["lens"] == res[1]["lens"]  # the tiny workload fixes its lengths
    assert res[0]["q"] != res[1]["q"]
    # The reference arm: one JSON line from rank 0, nothing from rank 1.
    lines = [l for l in res[0]["printed"].splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] == pytest.approx(1.5)
    assert line["n_gpus"] == 2 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert res[1]["printed"] == ""
