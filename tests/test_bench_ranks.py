"""bench.py's multi-process path on CPU: replicas over gloo, world size 2 (the data path
has no collective; only the timing reduction and the barrier do)."""

import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        # rank r "measured" 30 + 10 r microseconds per step on its replica
        ms = bench.max_over_ranks(torch, 0.030 + 0.010 * rank, world, "cpu")
        dist.barrier()
        results[rank] = (ms, bench.job_gbs(142_606_336, world, ms))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    world = 2
    mgr = mp.Manager()
    results = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), results), nprocs=world, join=True,
                       start_method="spawn")
    assert results[0] == results[1]
    ms, gbs = results[0]
    assert ms == pytest.approx(0.040)
    # both replicas' KV bytes over the slowest step time
    assert gbs == pytest.approx(2 * 142_606_336 / 40e-6 / 1e9)


def test_single_process_is_unchanged():
    import bench
    assert bench.max_over_ranks(torch, 0.0123, 1, "cpu") == 0.0123
    assert bench.job_gbs(1e9, 1, 1.0) == pytest.approx(1000.0)


def test_decode_source_hash_covers_the_decode_include_closure_only():
    # the DRAM-traffic rows are keyed by a hash of the decode kernels' sources: every decode
    # instantiation unit and header they include counts, the prefill kernels' headers do not
    import bench
    files = bench.decode_source_files()
    for name in ("kvq_decode_mma.cuh", "kvq_decode_hm.cuh", "kvq_encode.cuh", "mma_q8_0_q8_0.cu"):
        assert name in files
    for name in ("kvq_prefill.cuh", "kvq_prefill_tc.cuh", "kvq_tc.cuh", "prefill_pairs.cu"):
        assert name not in files
    assert len(bench.kernel_sources_sha()) == 16
