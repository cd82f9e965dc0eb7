"""bench.py's multi-rank host logic on CPU: two gloo ranks, max-over-ranks time
and whole-job throughput (no GPU)."""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    bench.dist_init(world, "gloo")
    local_time = 1.0 + rank            # rank 1 is the slow one
    t = bench.max_over_ranks(local_time)
    bench.barrier()
    q.put((rank, t, bench.job_throughput(1000, world, t), bench.dist_env()))
    dist.destroy_process_group()


def test_two_rank_max_and_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, thr, env in res:
        assert t == 2.0                       # max over ranks
        assert thr == pytest.approx(1000.0)   # 2 ranks x 1000 units / 2 s
        assert env == (rank, 2, rank)


def test_single_process_helpers():
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_throughput(4096, 1, 0.5) == 8192.0
    args = bench.parse_args([])
    assert args.gpus == 1 and args.warmup >= 3 and args.config == "finegrained_shared_bf16"


def test_dominant_kernel_flops():
    import moe_synth
    cfg = moe_synth.CONFIGS["mixtral_bf16"]
    stage, bound, flops, unit = bench.dominant_kernel(cfg)
    assert stage == "ffn_up" and bound == "tensor"
    assert flops == 2 * 4096 * 2 * 4096 * 14336 * 2


def test_dominant_kernel_fused_decode_bytes():
    """A small-batch layer run as one launch is measured on the whole layer's
    bytes: the selected experts' codes and scales once, the router's weights,
    x in and y out."""
    import moe_synth
    cfg = moe_synth.CONFIGS["gptoss_decode_mxfp4"].scaled(n=4)
    stage, bound, nbytes, unit = bench.dominant_kernel(cfg, active_experts=15, fused=True)
    assert (stage, bound, unit) == ("fused", "hbm", "GB/s")
    per_expert = 3 * (2880 * 2880 // 2 + 2880 * 2880 // 32)
    assert nbytes == 15 * per_expert + 128 * 2880 * 2 + 2 * 4 * 2880 * 2
    # the chained launches: the up-projection kernel
    stage, bound, _, _ = bench.dominant_kernel(cfg, active_experts=15)
    assert (stage, bound) == ("ffn_up", "hbm")
