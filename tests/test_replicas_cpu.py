"""The bench's N > 1 path on the host: two ranks over gloo on CPU.

With one process per GPU, each rank decodes its own B sequences (replicas,
weak scaling: the sequences are independent) with no collective on the data
path; the only cross-rank step is the max over ranks of the timings, and the
reference arm runs on rank 0 alone.  These tests run that host logic with two
gloo ranks.
"""
import argparse
import contextlib
import io
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    import rlt_inputs as ri
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = ri.preset("small")
        tok, prompt, acts = bench.rank_inputs(wl, rank)
        tok2, _, _ = bench.rank_inputs(wl, rank)
        # per-rank timings: the slowest rank must time the job
        t = [1.0 + rank, 2.0 - 0.5 * rank, 0.25 * (rank + 1)]
        tm = bench.max_over_ranks(t, world)
        dist.barrier()
        np.savez(os.path.join(out_dir, f"rank{rank}.npz"), tok=tok, acts=acts, same=np.array_equal(tok, tok2),
                 tmax=np.array(tm), value=bench.job_throughput(wl.B, wl.T, world, tm[0]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_sequences_and_take_the_slowest_time(tmp_path):
    import torch.multiprocessing as mp
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    r = [np.load(tmp_path / f"rank{i}.npz") for i in range(world)]
    # each rank's draw is deterministic and the ranks hold different sequences
    assert all(bool(x["same"]) for x in r)
    assert r[0]["tok"].shape == r[1]["tok"].shape
    assert not np.array_equal(r[0]["tok"], r[1]["tok"])
    # the teacher-forced actions are each rank's own next tokens
    for x in r:
        assert np.array_equal(x["acts"][:, :-1], x["tok"][:, 1:])
    # every rank sees the element-wise maximum over ranks
    expect = [2.0, 2.0, 0.5]
    for x in r:
        assert np.allclose(x["tmax"], expect)
    import rlt_inputs as ri
    wl = ri.preset("small")
    assert np.isclose(float(r[0]["value"]), wl.B * wl.T * world / 2.0)


def test_single_rank_reduction_is_identity():
    import bench
    assert bench.max_over_ranks([3.0, 1.0], 1) == [3.0, 1.0]


def test_reference_arm_runs_on_rank_zero_only():
    import bench
    args = argparse.Namespace(workload="tiny", steps=1, warmup=0, gpus=2)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(args, rank=1)
    assert buf.getvalue() == ""


def test_reference_arm_line_has_the_gpu_arms_keys():
    """The reference arm times the oracle on the host cores on the same
    workload config, metric and unit as the GPU arm."""
    import json
    import bench
    import rlt_inputs as ri
    args = argparse.Namespace(workload="tiny", steps=1, warmup=0, gpus=1)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(args, rank=0)
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["unit"] == bench.UNIT
    assert line["higher_is_better"] is True and line["value"] > 0
    assert line["config"] == bench.workload_config(ri.preset("tiny"), 1, 1)
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": bench.UNIT, "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
