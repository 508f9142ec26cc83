"""Host-side logic of the N > 1 benchmark path, on CPU with two gloo ranks.

The workload shards by batch with no exchange between ranks; what the ranks share is the
timing protocol: a barrier around the timed region, the maximum of the elapsed times over
ranks, and the whole-job throughput (all ranks' units over the slowest rank's time).
"""
from __future__ import annotations

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    r, w, local = bench.dist_env()
    assert (r, w, local) == (rank, world, rank)
    bench.dist_init(world, "gloo")
    try:
        bench.barrier(world)
        elapsed = 1.0 + rank                       # rank 1 is the slow one
        slowest = bench.allreduce_max(elapsed, world)
        rate = bench.aggregate_rate(100.0, world, slowest)
        bench.barrier(world)
        results[rank] = (slowest, rate)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_slowest_time_and_job_rate():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
        assert results[0] == results[1] == (2.0, 100.0)   # 2 ranks x 100 units / 2.0 s


def test_single_rank_helpers_are_identity():
    assert bench.allreduce_max(3.5, 1) == 3.5
    assert bench.aggregate_rate(10.0, 1, 2.0) == 5.0
    bench.barrier(1)


def test_code_hash_ignores_comments_and_layout_not_code():
    # the traffic record of profiles/ stays valid across comment edits, not code edits
    a = 'int x = 1; // note\n/* block\n comment */ int  y=2;\nconst char *s = "a // b";'
    b = 'int x=1;\nint y = 2; // other note\nconst char *s = "a // b";'
    assert bench.code_hash(a) == bench.code_hash(b)
    assert bench.code_hash(a) != bench.code_hash(a.replace("y=2", "y=3"))
    assert bench.code_hash(a) != bench.code_hash(a.replace('"a // b"', '"a "'))


def test_roofline_byte_and_flop_models():
    from linear_attention_recurrence_gdn_gb300.workloads import DECODE_B64, PREFILL_B4
    # 8 B per state element (read + write) dominates; the closed form of the bench's docstring
    assert bench.decode_bytes(DECODE_B64) == 271_073_792
    assert bench.scan_flops(PREFILL_B4) == 6 * 128 * 128 * 4 * 4096 * 32
    # bf16 block form: per warp and 16-token block 64 (X, Y) + 12 (d, O) + 32 (update) MMAs
    assert bench.scan_mma_flops(PREFILL_B4) == 4 * 32 * 8 * 108 * 4096 * 4096 // 16
    # Dk != Dv: X, Y run over Dk / 16 k-steps and the update over Dk / 8 n-tiles, on Dv / 16
    # warps: Dk = 64, Dv = 128 bf16 -> 32 + 12 + 16 MMAs on 8 warps; Dk = 128, Dv = 64 f16
    # (3 operand terms) -> 96 + 12 + 48 on 4 warps
    assert bench.scan_mma_flops(PREFILL_B4.replace(Dk=64)) == 4 * 32 * 8 * 60 * 4096 * 4096 // 16
    assert (bench.scan_mma_flops(PREFILL_B4.replace(Dv=64, act="f16"))
            == 4 * 32 * 4 * 156 * 4096 * 4096 // 16)
    # tensor-memory chunked kernel: per head and steady chunk 16x32 (tables) + 16x64 ([x|y])
    # + 12x32 (d, O) + 4x128 (update) + 6x64 (correction) = 2816 columns of 128x16 MMAs;
    # the first chunk has no cross table (8x32 fewer), the last no correction (6x64 fewer)
    assert bench.scan_tmem_mma_flops(PREFILL_B4) == 128 * (2 * 128 * 16) * (2816 * 128 - 640)


def test_reference_arm_prints_one_line(capsys):
    pytest.importorskip("numpy")
    rc = bench.main(["--impl", "reference", "--steps", "2", "--warmup", "3"])
    assert rc == 0
    import json
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
