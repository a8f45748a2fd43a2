"""Host-side logic of bench.py: FLOP counts, the whole-job aggregation over
ranks (world_size 2 over gloo on CPU), and the CPU-baseline sampler."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import bench
from exact_io_aware_30_gb300 import inputs, metrics


def test_workload_flops_match_the_closed_forms():
    w = inputs.workload(2)   # causal 8192: S(S+1)/2 pairs per head
    assert metrics.attention_flops(w) == 4.0 * 128 * 32 * (8192 * 8193 // 2)
    w = inputs.workload(4)   # no mask: S^2 pairs
    assert metrics.attention_flops(w) == 4.0 * 256 * 16 * 4096 * 4096
    w = inputs.workload(3)   # window 4096 over 18000 rows
    pairs = sum(min(i + 1, 4096) for i in range(18000))
    assert metrics.attention_flops(w) == 4.0 * 128 * 16 * pairs
    assert metrics.algorithmic_bytes(inputs.workload(0)) == 2 * 256 * 64 * 4 + 4 * 256


def test_whole_job_value_is_total_work_over_slowest_rank():
    assert bench.whole_job_value(1e12, 1, 1000.0) == pytest.approx(1.0)
    assert bench.whole_job_value(1e12, 4, 500.0) == pytest.approx(8.0)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [3.0, 5.0][rank]
    out[rank] = bench.reduce_max_time(ms, world)
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0] == 5.0 and out[1] == 5.0


def test_cpu_baseline_sampler_small():
    w = inputs.Workload("t", 1, 2, 300, 300, 64, inputs.BF16, "causal", seed=3)
    tf, cores, desc, dt = bench.cpu_oracle_sample(w, target_s=0.2)
    assert tf > 0 and cores >= 1 and "query rows" in desc


def test_recorded_traffic_requires_matching_source(tmp_path, monkeypatch):
    # a stale digest never yields a traffic figure
    assert bench.recorded_traffic("no_such_workload") is None


def test_recorded_decode_traffic_is_keyed_to_the_decode_sources():
    # the committed decode summary carries a traffic line for the one-row
    # workload; it is read only under the digest of the decode sources
    name = "decode_b128_h40_d128_bs16_ctx2048_fp16"
    summary = "fa_decode_gemv_kernel_launches_decode_b128_h40_d128_bs16_ctx2048_fp16.md"
    got = bench.recorded_traffic(name, summary, bench.DEC_SOURCES)
    text = open(os.path.join(bench.ROOT, "profiles", summary)).read()
    recorded = bench.kernel_source_digest(bench.DEC_SOURCES) in text
    assert (got is not None) == recorded
    if got is not None:
        assert got > 0
    # the forward's digest never matches it
    assert bench.recorded_traffic(name, summary) is None

