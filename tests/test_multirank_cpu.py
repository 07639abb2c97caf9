"""The N > 1 host logic of bench.py on CPU: two gloo ranks, each an independent
replica.  The job's time is the slowest rank's, its throughput counts every
rank's tokens, and the reduction is the only collective."""
import os
import socket
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
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 10.0 + 5.0 * rank          # rank 1 is the slow one
        job_ms = bench.max_over_ranks(local_ms, world, "cpu")
        value = bench.job_throughput(world, 16384, job_ms)
        out[rank] = (job_ms, value)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_count_all_tokens():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        assert all(p.exitcode == 0 for p in procs)
        res = dict(out)
    assert res[0] == res[1]                     # every rank agrees
    job_ms, value = res[0]
    assert job_ms == 15.0                       # the slowest rank sets the time
    assert value == pytest.approx(2 * 16384 / 15e-3)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(12.5, 1) == 12.5
    assert bench.job_throughput(1, 1000, 2.0) == pytest.approx(5e5)


def test_launches_per_step_by_workload():
    """The per-step launch count bench.py reports: three kernels for bf16, five
    when fwd_pass_state takes its two-pass form (long chains: at least 64
    chunks and at most half a chain per range), four for fp32."""
    sys.path.insert(0, ROOT)
    import bench
    from state_space_sequence_chunk_gb300 import synth
    W = synth.WORKLOADS
    assert bench.launches_per_step(W["mamba2_layer_bf16"], 152) == 3     # 16 chunks per chain
    assert bench.launches_per_step(W["short_streams_bf16"], 152) == 3    # 4 chunks per chain
    assert bench.launches_per_step(W["long_context_bf16"], 152) == 5     # 256 chunks, 12 chains
    assert bench.launches_per_step(W["tiny_fp32"], 152) == 4
    assert bench.launches_per_step(W["small_fp32"], 152) == 4


def test_cpu_baseline_reports_one_core_and_all_cores():
    """bench.py's cpu_baseline: the oracle on one core and on every core, each
    projected to the whole workload, with the thread count it used."""
    sys.path.insert(0, ROOT)
    import bench
    from state_space_sequence_chunk_gb300 import synth
    w = synth.WORKLOADS["tiny_fp32"]
    r = bench.cpu_baseline(w, synth.make_inputs(w), 0.5)
    assert r["kind"] == "oracle" and r["cores"] == 1 and r["value"] > 0
    assert r["all_cores"]["cores"] == (os.cpu_count() or 1) and r["all_cores"]["value"] > 0
