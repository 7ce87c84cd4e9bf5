"""Host-side logic of bench.py: max-over-ranks timing with two gloo ranks on the
CPU, the whole-job throughput formula, and the provenance check of the committed
ncu traffic figure."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(times[rank], dist)
        out[rank] = ms
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    times = [12.5, 31.25]
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, times, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1] == max(times)


def test_job_throughput_is_whole_job_weak_scaling():
    flops = 12 * 2048 * 20480 * 81920
    one = bench.job_throughput(flops, 10, 1, 300.0)
    assert one == pytest.approx(flops * 10 / 0.3 / 1e12)
    assert bench.job_throughput(flops, 10, 4, 300.0) == pytest.approx(4 * one)


def test_max_over_ranks_single_process_is_identity():
    assert bench.max_over_ranks(7.0, None) == 7.0


def test_traffic_figure_tracks_the_gemm_sources():
    value = bench.gemm_traffic_per_launch("mtnlg")
    assert value is None or value > 0
    assert bench.gemm_traffic_per_launch("tiny") is None


def test_gemm_hash_ignores_comments_only(tmp_path, monkeypatch):
    """The capture key changes with the GEMM code, not with its comments."""
    import shutil
    csrc = tmp_path / "transformer_lm_megatron_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name in bench.GEMM_SOURCES:
        shutil.copy(os.path.join(bench.ROOT, "transformer_lm_megatron_gb300", "csrc", name), csrc / name)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.gemm_source_hash()
    with open(csrc / "gemm_tc.cuh", "a") as fh:
        fh.write("\n// a comment\n\n")
    assert bench.gemm_source_hash() == h0
    with open(csrc / "gemm_tc.cuh", "a") as fh:
        fh.write("constexpr int kNotThere = 1;\n")
    assert bench.gemm_source_hash() != h0


def test_step_time_summary():
    s = bench.step_time_summary([3.0, 1.0, 2.0, 10.0])
    assert s == {"median": 2.5, "min": 1.0, "max": 10.0}
