"""Full-size parity: workloads 2-5 at their real sizes, generated on the device and run through the
same DropStep calls that bench.py times.  Every request is checked, not a sample:

* block scores of every request against the fp64 oracle (1e-3 relative; the oracle's inputs are
  regenerated on the host by the numpy generator, in a spawn process pool);
* the kept-block set of every request against the oracle's selection on the oracle's scores, with
  blocks within 1e-3 of the top-p threshold counted (UniPrefill section 3.3, Eq. 5);
* the selection on the GPU's own fp32 scores, bit-exact against the oracle's selection on those scores;
* the compaction (kept_index, query_start_loc, seq_lens, num_actual_tokens, drop history, positions,
  slots) bit-exact against the oracle's, and the WHOLE compacted hidden buffer bit-exact against the
  input rows it names (section 3.5, "vLLM scheduler integration");
* Eq. 8 (section 3.4) with new states that differ from the block input in every element: kept rows of
  the residual carry the new states, dropped rows stay byte-identical to the block input.
"""
import numpy as np
import pytest
import torch

import long_context_prefill_varlen_gb300 as up
import oracle
from synth import cpu as gen
from synth import gpu as sgpu
from synth import recipe
from tests import oracle_jobs, parity

pytestmark = pytest.mark.gpu

ROW_CHUNK = 1 << 16


def _bits(t):
    return t.view(torch.int16)


@pytest.mark.parametrize("cfg", [2, 3, 4, 5])
def test_fullsize_workload(cfg):
    w = recipe.workload(cfg)
    u = gen.mean_query_dirs(w)
    hot_tok = gen.hot_token_mask(w)
    # the oracle's scores of every request, on the host cores, started before any GPU work of this test
    ref_scores = oracle_jobs.all_block_scores(w, u, hot_tok)

    d = sgpu.build_device(w, u=u, hot_tok=hot_tok)
    # the device generator is the numpy generator's twin: spot-check a few rows of each tensor
    cu = np.asarray(w.cu_seqlens())
    for t in (0, int(cu[-1]) // 2, int(cu[-1]) - 3):
        assert np.array_equal(_bits(d["K"][t:t + 3]).cpu().numpy().view(np.uint16), gen.gen_k(w, t, t + 3, u, hot_tok))
        assert np.array_equal(_bits(d["hidden"][t:t + 3]).cpu().numpy().view(np.uint16), gen.gen_hidden(w, t, t + 3))

    step = up.DropStep(d["cu_seqlens"], w.T, w.Hq, w.Hkv, w.dk, w.hdim, G=w.G, n=w.n, A=w.A, p=w.p, L=2, layer=0)
    step.score(d["Q"], d["K"])
    step.select()
    step.compact(d["hidden"], d["positions"], d["slots"])
    # Eq. 8 with sublayers that change every element: the compacted rows with their lowest bit flipped
    new_states = (_bits(step.out_hidden) ^ 1).view(torch.bfloat16)
    residual = d["hidden"].clone()
    step.scatter_back(new_states, residual)
    torch.cuda.synchronize()
    step.check()

    cb = oracle.cu_blocks_of(cu, w.G)
    bs = step.block_scores.cpu().numpy()[:cb[-1]]
    bk = step.block_keep.cpu().numpy()[:cb[-1]]
    tk = step.token_keep.cpu().numpy()
    ks = step.kstar.cpu().numpy()

    # scores and kept sets of every request against the oracle
    boundary, max_rel = 0, 0.0
    for r in range(w.R):
        ref = ref_scores[r]
        max_rel = max(max_rel, parity.check_block_scores(bs[cb[r]:cb[r + 1]], ref))
        boundary += parity.check_selection(bk[cb[r]:cb[r + 1]], tk[cu[r]:cu[r + 1]], ref, [0, cu[r + 1] - cu[r]],
                                           w.G, w.n, w.A, w.p)
    # selection on the GPU's own scores: bit-exact
    sel = oracle.select(bs.astype(np.float32).astype(np.float64), cu, w.G, w.n, w.A, w.p)
    assert np.array_equal(tk, sel["token_keep"])
    assert np.array_equal(bk, sel["block_keep"])
    assert np.array_equal(ks, sel["kstar"])

    # compaction and metadata, bit-exact given the GPU's mask
    ref = oracle.compact(tk, cu)
    Tp = ref["num_actual_tokens"]
    assert int(step.num_actual.item()) == Tp
    ki = step.kept_index.cpu().numpy()[:Tp]
    assert np.array_equal(ki, ref["kept_index"])
    assert np.array_equal(step.new_cu.cpu().numpy(), ref["new_cu_seqlens"])
    assert np.array_equal(step.new_len.cpu().numpy(), ref["seq_lens"])
    assert np.array_equal(step.kept_len.cpu().numpy()[0], ref["seq_lens"])
    assert step.drop_layer.cpu().numpy()[0] == 1
    assert np.array_equal(step.out_positions.cpu().numpy()[:Tp], gen.gen_positions(w)[ki])
    assert np.array_equal(step.out_slots.cpu().numpy()[:Tp], gen.gen_slots(w)[ki])

    # the whole compacted hidden buffer against the input rows it names, and Eq. 8 over the whole residual
    ref_idx = torch.from_numpy(ref["kept_index"]).to(d["hidden"].device)
    hid = _bits(d["hidden"])
    for k0 in range(0, Tp, ROW_CHUNK):
        k1 = min(Tp, k0 + ROW_CHUNK)
        rows = hid.index_select(0, ref_idx[k0:k1])
        assert torch.equal(_bits(step.out_hidden[k0:k1]), rows), f"compacted rows {k0}..{k1}"
        assert torch.equal(_bits(residual).index_select(0, ref_idx[k0:k1]), rows ^ 1), f"Eq. 8 kept rows {k0}..{k1}"
    dropped = torch.ones(w.T, dtype=torch.bool, device=hid.device)
    dropped[ref_idx] = False
    dropped_idx = torch.nonzero(dropped).flatten()
    assert dropped_idx.numel() == w.T - Tp
    for k0 in range(0, dropped_idx.numel(), ROW_CHUNK):
        sel_rows = dropped_idx[k0:k0 + ROW_CHUNK]
        assert torch.equal(_bits(residual).index_select(0, sel_rows), hid.index_select(0, sel_rows)), "Eq. 8 dropped rows"
    print(f"config {cfg}: T={w.T} T'={Tp} rho={Tp / w.T:.4f} requests={w.R} blocks={int(cb[-1])} "
          f"max rel score err={max_rel:.2e} boundary blocks={boundary}")
