"""The benchmark's multi-rank bookkeeping on CPU with two gloo ranks: every
rank runs its own replica, times are reduced with a max over ranks, and the
headline value counts the work of all ranks."""
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [3.0, 5.0][rank]
    got = bench.reduce_max(ms, world, torch.device("cpu"))
    out[rank] = got
    dist.barrier()
    dist.destroy_process_group()


def test_reduce_max_two_ranks():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    assert out[0] == 5.0 and out[1] == 5.0


def test_rate_and_work_accounting():
    w = bench.inputs.WORKLOADS["gqa_prefill"]
    # 4 sequences x 32 heads x 4096*4097/2 pairs
    assert bench.allowed_pairs(w) == 4 * 32 * 4096 * 4097 // 2
    assert bench.fwd_flops(w) == 4.0 * 128 * bench.allowed_pairs(w)
    d = bench.inputs.WORKLOADS["decode_q1"]
    assert bench.allowed_pairs(d) == 32 * 32 * 32768
    assert bench.decode_bytes(d) == 2 * 32 * 32768 * 8 * 128 * 2 + 2 * 32 * 32 * 128 * 2 + 32 * 32 * 4
    e = bench.inputs.WORKLOADS["decode_empty_rows"]
    assert bench.allowed_pairs(e) == 32 * 32 * 528
    # two ranks doing the same work at the slowest rank's time
    assert bench.rate(2 * 1e12, "TFLOP/s", 1000.0) == pytest.approx(2.0)
    assert bench.count_kernels("fwd_tc_d128_packgqa grid=(1,8,512) tile_tokens=32 splits=16 +combine") == 2
    assert bench.count_kernels("bwd_pre+bwd_dq_simt+bwd_dkdv_simt_bf16_d128") == 3
