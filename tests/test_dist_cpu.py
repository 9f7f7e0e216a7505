"""Multi-rank host logic on CPU (gloo, world size 2): the tensor-parallel
amax MAX-reduce gives every rank the amax -- and so the scale -- of the
whole tensor, bit for bit; and the step-time reduction takes the max over
ranks."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
import synthetic


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from scaled_fp8_linear_gb300.distributed import max_over_ranks, sync_amax
        W = synthetic.student_t((512, 256), 3, 0.02, seed=42)
        shard = W[rank * 256:(rank + 1) * 256]            # TP split of the output rows
        bits = synthetic.bf16_bits(shard)
        local = torch.tensor([float(oracle.amax(bits))], dtype=torch.float32)
        sync_amax(local)
        st = oracle.ScaleState(16)
        oracle.update_scale(st, local.item(), oracle.ALGO_MAX, oracle.E4M3)
        t = max_over_ranks(10.0 + rank)
        q.put((rank, local.item(), float(st.scale[0]), t))
    finally:
        dist.destroy_process_group()


def test_tp_amax_sync_and_time_reduction_two_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    W = synthetic.student_t((512, 256), 3, 0.02, seed=42)
    full = oracle.amax(synthetic.bf16_bits(W))
    st = oracle.ScaleState(16)
    oracle.update_scale(st, full, oracle.ALGO_MAX, oracle.E4M3)
    for rank, amax, scale, t in out:
        assert np.float32(amax) == full
        assert np.float32(scale) == st.scale[0]
        assert t == 11.0
