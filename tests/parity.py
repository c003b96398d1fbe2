"""Comparison of the CUDA path with the fp64 oracle, with the tolerances of the drop step.

* block scores: |gpu - oracle| <= 1e-3 * oracle (+1e-12 absolute), fp32 accumulation from bf16;
* kept blocks: identical, except blocks whose oracle score lies within 1e-3 relative of the
  top-p threshold tau (the oracle score of the k*-th ranked block); such blocks are counted;
* compaction, metadata, scatter-back: bit-exact given the GPU's own keep mask.
"""
from __future__ import annotations

import numpy as np

import oracle

RTOL_SCORE = 1e-3
RTOL_THRESHOLD = 1e-3


def bf16_to_f64(t):
    """torch bf16 tensor (any device) -> numpy fp64 (bf16 -> fp32 widening is exact)."""
    return t.detach().float().cpu().numpy().astype(np.float64)


def check_block_scores(gpu, ref, rtol=RTOL_SCORE):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape
    err = np.abs(gpu - ref)
    bad = err > rtol * np.abs(ref) + 1e-12
    rel = float(np.max(err / np.maximum(np.abs(ref), 1e-30))) if len(ref) else 0.0
    assert not bad.any(), f"{int(bad.sum())} block scores off by more than {rtol} relative (max rel {rel:.3e})"
    return rel


def check_selection(gpu_block_keep, gpu_token_keep, ref_scores, cu_seqlens, G, n, A, p, rtol=RTOL_THRESHOLD):
    """GPU keep masks against the oracle's selection on the oracle's scores; returns #boundary blocks."""
    cu = [int(c) for c in cu_seqlens]
    cb = oracle.cu_blocks_of(cu, G)
    boundary = 0
    gbk = np.asarray(gpu_block_keep).astype(bool)
    gtk = np.asarray(gpu_token_keep).astype(bool)
    for r in range(len(cu) - 1):
        N = cu[r + 1] - cu[r]
        if N == 0:
            continue
        b = np.asarray(ref_scores[cb[r]:cb[r + 1]], dtype=np.float64)
        d = oracle.select_request(b, N, G, n, A, p)
        tau = b[d["order"][d["kstar"] - 1]]
        diff = np.flatnonzero(gbk[cb[r]:cb[r + 1]] != d["block_keep"])
        for g in diff:
            assert abs(b[g] - tau) <= rtol * tau, (
                f"request {r} block {g}: score {b[g]:.6e} is not within {rtol} of the threshold {tau:.6e}")
        boundary += len(diff)
        # the token mask is the block decision lifted to tokens, plus the forced tokens
        i = np.arange(N)
        tk = gtk[cu[r]:cu[r + 1]]
        bk = gbk[cb[r]:cb[r + 1]]
        forced_tok = (i < A) | (i >= N - n)
        assert np.all(tk[forced_tok])
        forced_blk = np.array([(g * G < A) or ((g + 1) * G > N - n) for g in range(len(b))], dtype=bool)
        blk = i // G
        plain = ~forced_blk[blk]
        assert np.array_equal(tk[plain], bk[blk[plain]])
        for g in np.flatnonzero(forced_blk):           # non-forced tokens of a forced block share one decision
            sel = (blk == g) & ~forced_tok
            if sel.any():
                assert tk[sel].all() or not tk[sel].any()
        assert np.array_equal(bk, np.array([tk[blk == g].any() for g in range(len(b))]))
    return boundary


def check_compaction(gpu, token_keep, cu_seqlens, hidden=None, positions=None, slots=None, L=None, layer=None):
    """gpu: dict of numpy arrays from the CUDA path; everything bit-exact against oracle.compact."""
    ref = oracle.compact(token_keep, cu_seqlens, hidden, positions, slots)
    Tp = ref["num_actual_tokens"]
    assert int(gpu["num_actual"]) == Tp
    assert np.array_equal(gpu["kept_index"][:Tp], ref["kept_index"])
    assert np.array_equal(gpu["new_cu"], ref["new_cu_seqlens"])
    assert np.array_equal(gpu["new_len"], ref["seq_lens"])
    if hidden is not None:
        assert np.array_equal(gpu["out_hidden"][:Tp], ref["hidden"])
    if positions is not None:
        assert np.array_equal(gpu["out_positions"][:Tp], ref["positions"])
    if slots is not None:
        assert np.array_equal(gpu["out_slots"][:Tp], ref["slots"])
    if layer is not None:
        assert np.array_equal(gpu["kept_len"][layer], ref["seq_lens"])
        assert gpu["drop_layer"][layer] == 1
    return Tp


def step_to_numpy(step, with_hidden=True):
    import torch
    out = dict(block_scores=step.block_scores.cpu().numpy(), block_keep=step.block_keep.cpu().numpy(),
               token_keep=step.token_keep.cpu().numpy(), kstar=step.kstar.cpu().numpy(),
               kept_index=step.kept_index.cpu().numpy(), new_cu=step.new_cu.cpu().numpy(),
               new_len=step.new_len.cpu().numpy(), num_actual=int(step.num_actual.item()),
               kept_len=step.kept_len.cpu().numpy(), drop_layer=step.drop_layer.cpu().numpy(),
               out_positions=step.out_positions.cpu().numpy(), out_slots=step.out_slots.cpu().numpy())
    if with_hidden and step.out_hidden is not None:
        out["out_hidden"] = step.out_hidden.cpu().view(torch.int16).numpy().view(np.uint16)
    if step.token_scores is not None:
        out["token_scores"] = step.token_scores.cpu().numpy()
    return out
