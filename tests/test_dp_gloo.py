"""Data parallelism over two CPU ranks (gloo): each rank computes the oracle's gradients
on its half of the batch and the ranks average them with one all-reduce; the result
equals the full-batch gradient.  This is the single exchange a multi-GPU version of the
training step would add after the backward pass (every run of the CUDA library here has
one GPU, so the library itself has no collective)."""
import os
import socket

import numpy as np
import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_path):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import torch
    import torch.distributed as dist
    from step_gpt_train_03_b300 import synth
    from tests.oracle_helpers import make_oracle
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    tokens, targets = synth.uniform_tokens(512, 4, 32, 9)
    shard = slice(rank * 2, rank * 2 + 2)
    o = make_oracle(synth.TINY, 3)
    loss = o.forward(tokens[shard], targets[shard])
    o.zero_grad()
    o.backward()
    g = torch.from_numpy(o.flat_grad.copy())
    dist.all_reduce(g, op=dist.ReduceOp.SUM)
    g /= world
    lt = torch.tensor([loss], dtype=torch.float64)
    dist.all_reduce(lt, op=dist.ReduceOp.SUM)
    if rank == 0:
        np.save(out_path, g.numpy())
        np.save(out_path + ".loss.npy", (lt / world).numpy())
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_gradient_average_equals_full_batch(tmp_path):
    import torch.multiprocessing as mp
    from step_gpt_train_03_b300 import synth
    from tests.oracle_helpers import make_oracle, rel_max_err
    out = str(tmp_path / "g.npy")
    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
    g_dp = np.load(out)
    loss_dp = float(np.load(out + ".loss.npy")[0])
    tokens, targets = synth.uniform_tokens(512, 4, 32, 9)
    full = make_oracle(synth.TINY, 3)
    loss = full.forward(tokens, targets)
    full.zero_grad()
    full.backward()
    assert rel_max_err(g_dp, full.flat_grad) < 1e-12
    assert abs(loss_dp - loss) < 1e-12
