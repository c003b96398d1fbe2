"""Per-request oracle jobs for a process pool (started with the 'spawn' method).

A job regenerates one request's inputs with the numpy input generator (synth.cpu) and runs the fp64
oracle on them, so the oracle side of the full-size parity tests touches no CUDA code at all.  This
module imports only numpy, the oracle and the CPU generator, so that a spawned worker starts quickly.
"""
from __future__ import annotations

import os

import numpy as np

import oracle
from synth import cpu as gen


def request_block_scores(args):
    """fp64 block scores (Eqs. 2-4) of request r of workload w; u and hot_tok as from synth.cpu."""
    w, r, u, hot_tok = args
    cu = w.cu_seqlens()
    a, b = cu[r], cu[r + 1]
    N = b - a
    if N == 0:
        return r, np.zeros(0)
    ne = min(w.n, N)
    Q = np.zeros((N, w.Hq, w.dk))
    Q[N - ne:] = gen.bf16_bits_to_f32(gen.gen_q(w, b - ne, b))
    K = gen.bf16_bits_to_f32(gen.gen_k(w, a, b, u, hot_tok)).astype(np.float64)
    return r, oracle.block_scores(Q, K, [0, N], w.G, w.n)


def all_block_scores(w, u, hot_tok, requests=None):
    """Oracle block scores of the given requests (default: all) of w, computed in parallel on the host
    cores; returns {r: fp64 array}.  Longest requests are submitted first."""
    import multiprocessing as mp
    requests = list(range(w.R)) if requests is None else list(requests)
    requests.sort(key=lambda r: -w.lengths[r])
    try:
        cores = len(os.sched_getaffinity(0))
    except AttributeError:
        cores = os.cpu_count() or 1
    procs = max(1, min(len(requests), cores // 2 if cores >= 4 else 1))
    threads = max(1, cores // procs)
    env = {k: str(threads) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    saved = {k: os.environ.get(k) for k in env}
    os.environ.update(env)                     # inherited by the spawned workers' BLAS
    try:
        with mp.get_context("spawn").Pool(procs) as pool:
            out = dict(pool.imap_unordered(request_block_scores, [(w, r, u, hot_tok) for r in requests]))
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    return out
