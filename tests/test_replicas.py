"""The N>1 bench path runs independent replicas (weak scaling): each rank
times its own stack, the ranks meet only at the host barriers, and the job's
throughput is every rank's tokens over the slowest rank's time.  Checked
here with world_size-2 gloo process groups on the CPU."""
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        local_ms = [12.5, 20.0][rank]
        ms, value = bench.job_throughput(local_ms, units_per_rank=30, pg=dist, device="cpu")
        out[rank] = (ms, value)
    finally:
        dist.destroy_process_group()


def test_job_throughput_takes_slowest_rank_and_all_units():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        ms, value = out[r]
        assert ms == 20.0
        assert value == pytest.approx(2 * 30 / 0.020)


def test_job_throughput_single_rank():
    sys.path.insert(0, ROOT)
    import bench
    ms, value = bench.job_throughput(8.0, units_per_rank=4)
    assert ms == 8.0 and value == pytest.approx(500.0)


def test_reference_arm_prints_only_on_rank_0():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "0"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_replicas_draw_distinct_inputs():
    sys.path.insert(0, ROOT)
    from moe_decode_layer_gemv_gb300 import synth
    w = synth.STACK
    seed = 0
    # the bench offsets each rank's seed by 7919 * rank
    x0 = synth.make_x(w, 0, seed=seed, device="cpu")
    x1 = synth.make_x(w, 0, seed=seed + 7919, device="cpu")
    assert not torch.equal(x0, x1)
