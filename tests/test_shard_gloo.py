"""The multi-GPU path's host logic on two gloo ranks (CPU): request sharding and the global metadata.

Each rank runs the oracle's drop step on its own requests only (the kernels are request-local, so a
rank needs no other rank's data); the global query_start_loc rebuilt from the per-rank kept lengths
must equal the unsharded oracle's, and the per-rank kept sets must be the unsharded ones.
"""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from long_context_prefill_varlen_gb300 import shard
from synth import cpu as gen
from synth import recipe

LENGTHS = (700, 129, 2000, 64, 0, 1500, 300)


def _workload():
    return recipe.small(lengths=LENGTHS, Hq=4, Hkv=2, dk=64, hdim=16, G=64, n=128, A=128, p=0.9,
                        hot=("frac", 0.2), salt=71)


def _oracle_step(host, cu, w):
    Q = gen.bf16_bits_to_f32(host["Q"]).astype(np.float64)
    K = gen.bf16_bits_to_f32(host["K"]).astype(np.float64)
    return oracle.drop_step(Q, K, cu, w.G, w.n, w.A, w.p)


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = _workload()
        host = gen.materialize(w, with_hidden=False)
        gcu = w.cu_seqlens()
        mine, lcu = shard.local_requests(LENGTHS, world, rank)
        # this rank's packed inputs: its requests' rows only
        rows = np.concatenate([np.arange(gcu[r], gcu[r + 1]) for r in mine]) if mine else np.zeros(0, int)
        local = dict(Q=host["Q"][rows], K=host["K"][rows])
        out = _oracle_step(local, lcu, w)
        kept = out["compact"]["seq_lens"]
        qsl = shard.global_query_start_loc(LENGTHS, kept, world, rank)
        q.put((rank, mine, out["token_keep"].tolist(), qsl.tolist()))
    finally:
        dist.destroy_process_group()


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def test_assignment_is_balanced_and_complete():
    owner = shard.assign_requests(LENGTHS, 2)
    assert sorted(set(owner)) == [0, 1]
    loads = [sum(L for L, o in zip(LENGTHS, owner) if o == k) for k in range(2)]
    assert abs(loads[0] - loads[1]) <= max(LENGTHS)
    assert shard.assign_requests(LENGTHS, 2) == owner          # deterministic


def test_two_gloo_ranks_reproduce_the_unsharded_step():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=240) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    w = _workload()
    host = gen.materialize(w, with_hidden=False)
    ref = _oracle_step(host, w.cu_seqlens(), w)
    gcu = w.cu_seqlens()
    qsls = [r[3] for r in res]
    assert qsls[0] == qsls[1] == ref["compact"]["new_cu_seqlens"].tolist()
    for rank, mine, tk, _ in res:                               # per-rank masks are the unsharded ones
        expect = np.concatenate([ref["token_keep"][gcu[r]:gcu[r + 1]] for r in mine]) if mine else []
        assert list(tk) == list(expect)
