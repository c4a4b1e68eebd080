"""The N > 1 host logic on CPU with gloo ranks: loads summed across replicas
give every rank the bias update of the global batch, bit-for-bit equal to a
single process that routed all tokens; mismatched ranks and a missing rank
raise instead of producing a wrong bias."""
import datetime
import multiprocessing as mp
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist

from expert_ffn_layer_affinity_b300 import synth
from expert_ffn_layer_affinity_b300.dist import allreduce_loads
from oracle import moe_ref as ref

T, E, K, GAMMA = 512, 64, 6, 1e-3


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, world, port, timeout_s=20):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=timeout_s))


def _replica(rank, world, port, q):
    _init(rank, world, port)
    b = np.zeros(E, dtype=np.float32)
    for step in range(3):
        s = synth.make_affinities(T, E, step=step * world + rank, seed=3, skew=0.05)
        idx, _ = ref.select_experts(s.numpy(), b, K)
        load = torch.from_numpy(ref.expert_load(idx, E))
        n = allreduce_loads(load)
        b = ref.bias_update(load.numpy(), b, T * n, K, E, GAMMA)
    q.put((rank, b.view(np.uint32).copy()))
    dist.destroy_process_group()


def _mismatch(rank, world, port, q):
    _init(rank, world, port)
    load = torch.zeros(E + rank, dtype=torch.int32)
    try:
        allreduce_loads(load)
        q.put((rank, "no error"))
    except ValueError as e:
        q.put((rank, "ValueError"))
    dist.destroy_process_group()


def _lonely(rank, world, port, q):
    try:
        _init(rank, world, port, timeout_s=3)
        allreduce_loads(torch.zeros(E, dtype=torch.int32))
        q.put((rank, "no error"))
    except Exception as e:  # the peer never joins
        q.put((rank, type(e).__name__))


def run(target, world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=target, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
    return out


def test_two_replicas_match_single_process():
    out = run(_replica, 2)
    assert np.array_equal(out[0], out[1])
    b = np.zeros(E, dtype=np.float32)
    for step in range(3):
        s = torch.cat([synth.make_affinities(T, E, step=step * 2 + r, seed=3, skew=0.05)
                       for r in range(2)])
        idx, _ = ref.select_experts(s.numpy(), b, K)
        b = ref.bias_update(ref.expert_load(idx, E), b, 2 * T, K, E, GAMMA)
    assert np.array_equal(out[0], b.view(np.uint32))


def test_mismatched_expert_counts_raise_on_every_rank():
    out = run(_mismatch, 2)
    assert out == {0: "ValueError", 1: "ValueError"}


def test_missing_rank_times_out_with_an_error():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    p = ctx.Process(target=_lonely, args=(0, 2, free_port(), q))
    p.start()
    rank, err = q.get(timeout=120)
    p.join(timeout=60)
    assert err != "no error"
