"""The multi-rank host logic of the bench, as two gloo ranks on the CPU.

The decode step shards as replicas: each rank decodes its own batch of
sequences and no data crosses ranks.  The ranks meet only to time the job:
a barrier on both sides of the timed region, then the slowest rank's time,
which every rank receives.  Rank 0 alone prints.  These tests run that logic
with two processes and check that per-rank results equal what one process
computes for the same seeds (so no exchange step is missing).
"""
import contextlib
import io
import json
import os
import socket
import sys
import tempfile

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

TINY = dict(name="tiny_bf16_b2_s40", dtype="bf16", batch=2, heads=16, s_max=40, hidden=2048)


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _replica_output(seed: int):
    """Oracle output of one rank's replica (the tiny workload drawn from `seed`)."""
    from oracle import mla_oracle as O
    from workloads import MlaConfig, make_inputs
    cfg = MlaConfig(**TINY)
    a = make_inputs(cfg, seed=seed).as_float64_numpy()
    r = O.decode_absorbed(a["q_nope"], a["q_rope"], a["w_uk"], a["w_uv"], a["cache"],
                          a["lengths"], a["positions"], cfg.softmax_scale, cfg.rope_base)
    return r["o"]


def _rank_main(rank, world, port, outdir):
    sys.path.insert(0, ROOT)
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    import bench
    res = {}
    dist.barrier()
    # the slowest rank's time reaches every rank
    my_ms = 10.0 + 5.0 * rank
    res["max_ms"] = bench.max_over_ranks(my_ms, torch.device("cpu"), world)
    # whole-job throughput: units of all ranks over the slowest rank's time
    res["rate"] = bench.whole_job_rate(1000.0, 4, world, res["max_ms"] / 1e3)
    # each rank decodes its own replica; gather the outputs only to check them
    o = torch.from_numpy(_replica_output(seed=rank))
    gathered = [torch.empty_like(o) for _ in range(world)]
    dist.all_gather(gathered, o)
    res["gathered"] = [g.tolist() for g in gathered]
    # the reference arm: only rank 0 works and prints
    args = bench.parse(["--impl", "reference", "--steps", "1", "--warmup", "0",
                        "--gpus", str(world), "--workload", "v2lite_f32_b1_s64"])
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = bench.main_with(args, rank=rank, world=world)
    res["ref_rc"] = rc
    res["ref_out"] = buf.getvalue()
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(outdir, f"rank{rank}.json"), "w") as f:
        json.dump(res, f)


def test_two_gloo_ranks_time_and_shard_as_replicas():
    world = 2
    port = _free_port()
    with tempfile.TemporaryDirectory() as d:
        mp.start_processes(_rank_main, args=(world, port, d), nprocs=world, join=True,
                           start_method="spawn")
        res = [json.load(open(os.path.join(d, f"rank{r}.json"))) for r in range(world)]
    for r in res:
        assert r["max_ms"] == 15.0
        assert r["rate"] == pytest.approx(1000.0 * 4 * 2 / 0.015)
        assert r["ref_rc"] == 0
    # replicas: what rank r computed equals a single-process run of seed r
    for r in range(world):
        np.testing.assert_array_equal(np.array(res[0]["gathered"][r]), _replica_output(seed=r))
    # the two replicas are different work, not copies
    assert not np.allclose(res[0]["gathered"][0], res[0]["gathered"][1])
    # rank 0 printed exactly one reference line; rank 1 printed nothing
    lines = [l for l in res[0]["ref_out"].splitlines() if l.strip()]
    assert len(lines) == 1 and json.loads(lines[0])["impl"] == "reference"
    assert res[1]["ref_out"].strip() == ""


def test_single_rank_helpers_need_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, torch.device("cpu"), 1) == 3.5
    assert bench.whole_job_rate(10.0, 3, 1, 2.0) == 15.0
