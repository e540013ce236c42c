"""World-size-2 replica path on CPU (gloo): each rank runs the oracle generation loop on
its own block of sequences; the gathered outputs equal one process running both blocks
(sequences never interact), and the timing reduction takes the slowest rank."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import fg_synth
from bit_compressed_throughput_gb300 import replicas

WL = fg_synth.WORKLOADS["tiny"].with_(h=128, H=2, d=64, f=128, s=4, n=3, g=1, m=2, L=1)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _run_block(rank):
    import oracle
    params = fg_synth.layer_params(WL, 0, random_affine=True)
    layers = [oracle.QuantLayer(params, WL.H, WL.d, WL.ln_eps)]
    seqs = replicas.block_sequences(rank, WL.B)
    out = oracle.run_stack(layers, fg_synth.prompt_states(WL, seqs),
                           fg_synth.step_states(WL, seqs), cap=WL.cap)
    return out["steps"]                     # [n-1][B][h]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    steps = torch.from_numpy(_run_block(rank))
    gathered = [torch.zeros_like(steps) for _ in range(world)]
    dist.all_gather(gathered, steps)
    slowest = replicas.max_over_ranks(10.0 + rank, dist)
    if rank == 0:
        q.put((torch.cat(gathered, dim=1).numpy(), slowest))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_replicas_match_single_process():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    gathered, slowest = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    import oracle
    params = fg_synth.layer_params(WL, 0, random_affine=True)
    layers = [oracle.QuantLayer(params, WL.H, WL.d, WL.ln_eps)]
    seqs = np.arange(2 * WL.B)
    ref = oracle.run_stack(layers, fg_synth.prompt_states(WL, seqs),
                           fg_synth.step_states(WL, seqs), cap=WL.cap)["steps"]
    assert np.array_equal(gathered, ref)
    assert slowest == 11.0
    assert replicas.total_tokens(2, WL.B, WL.n, 5) == 2 * WL.B * WL.n * 5
