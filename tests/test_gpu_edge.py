"""Varlen edges of the whole drop step on the GPU (through DropStep and the C ABI): hundreds of tiny
requests mixed with a few long ones (empty requests, requests shorter than one block, than the window,
than the sinks), and a batch with no tokens at all."""
import numpy as np
import pytest
import torch

import long_context_prefill_varlen_gb300 as up
import oracle
from synth import cpu as gen
from synth import gpu as sgpu
from synth import recipe
from tests import parity

pytestmark = pytest.mark.gpu


def _run(w, L=2, layer=1):
    host = gen.materialize(w)
    d = sgpu.to_device(host)
    step = up.DropStep(d["cu_seqlens"], w.T, w.Hq, w.Hkv, w.dk, w.hdim, G=w.G, n=w.n, A=w.A, p=w.p, L=L,
                       layer=layer)
    resid = d["hidden"].clone()
    step.run(d["Q"], d["K"], d["hidden"], d["positions"], d["slots"], residual=resid)
    torch.cuda.synchronize()
    step.check()
    return host, step, resid


def test_hundreds_of_tiny_requests_among_long_ones():
    """600 requests of 0-70 tokens around three of 900-2600 tokens: the work items, the per-request
    selection CTAs and the compaction tiles all cross many request boundaries."""
    rng = np.random.default_rng(600)
    lengths = [int(x) for x in rng.integers(0, 71, 600)]
    for pos, L in ((17, 2600), (300, 900), (599, 1300)):
        lengths[pos] = L
    w = recipe.small(lengths=tuple(lengths), Hq=8, Hkv=2, dk=128, hdim=64, G=32, n=32, A=16, p=0.9,
                     hot=("frac", 0.2), salt=600)
    host, step, resid = _run(w)
    got = parity.step_to_numpy(step)
    Q = gen.bf16_bits_to_f32(host["Q"]).astype(np.float64)
    K = gen.bf16_bits_to_f32(host["K"]).astype(np.float64)
    ref = oracle.block_scores(Q, K, host["cu_seqlens"], w.G, w.n)
    parity.check_block_scores(got["block_scores"][:len(ref)], ref)
    parity.check_selection(got["block_keep"][:len(ref)], got["token_keep"], ref, host["cu_seqlens"], w.G, w.n, w.A,
                           w.p)
    parity.check_compaction(got, got["token_keep"], host["cu_seqlens"], host["hidden"], host["positions"],
                            host["slots"], layer=1)
    assert np.array_equal(resid.cpu().view(torch.int16).numpy().view(np.uint16), host["hidden"])
    # empty requests keep nothing, requests within the sinks and the window keep everything
    cu = host["cu_seqlens"]
    kept = got["new_len"]
    for r, L in enumerate(lengths):
        if L <= w.A + w.n:
            assert kept[r] == L, (r, L, kept[r])


def test_a_batch_without_tokens():
    """Three empty requests (T = 0): every call runs, nothing is kept, the metadata is all zeros."""
    w = recipe.small(lengths=(0, 0, 0), Hq=4, Hkv=2, dk=128, hdim=64, G=64, n=128, salt=3)
    host, step, _ = _run(w)
    assert int(step.num_actual.item()) == 0
    assert np.array_equal(step.new_cu.cpu().numpy(), np.zeros(4, dtype=np.int32))
    assert np.array_equal(step.new_len.cpu().numpy(), np.zeros(3, dtype=np.int32))
    assert np.array_equal(step.kstar.cpu().numpy(), np.zeros(3, dtype=np.int32))
    assert np.array_equal(step.kept_len.cpu().numpy()[1], np.zeros(3, dtype=np.int32))
    assert int(step.drop_layer.cpu().numpy()[1]) == 1
